"""Benchmark of the W4A16 INT4 MoE expert GEMM pair on one GB300.

Metric (the pages' method: per-layer time of the gate_up GEMM plus the down
GEMM, routing and activation excluded; page "vLLM 宣布 Humming 后端可运行 …
Chord 内核 …", section "六个场景的逐层测量与限定条件"): microseconds per
layer, lower is better, plus achieved HBM GB/s and TFLOP/s against the
measured roofline.

One step = one decode step through `--layers` MoE layers of the headline
shard shape (EP8 decode by default): per layer routing alignment, gate_up,
silu_and_mul and down over the same batch. Before every layer L2 is flushed
(a 256 MiB write), so each layer streams its 1.19 GB of weights from HBM as a
distinct layer would. The reported value is the mean over all timed layers
of the CUDA-event time of gate_up plus down, with inputs already resident in
HBM.

The same run then measures every other configuration of the shard shapes
(TP8 T=16/64/256, EP8 prefill, grouped contiguous 128 and 1024 rows per
expert, grouped masked with a 32-row budget) and reports them in the
`configs` object of the JSON line, each with its roofline fraction against
the bound that applies (HBM for the weight-bound shapes, BF16 tensor peak for
the compute-bound ones).

`--impl reference` times the float64 CPU oracle on the host cores instead:
each step one whole layer of the same workload (every active expert, all its
routed rows).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                       [--layers L] [--no-configs]
                       [--workload ep8_decode|ep8_decode_e12|tp8_16|tp8_64|tp8_256|ep8_prefill|ep8_prefill_x4|tiny
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
# nominal GB300 figures, reported beside the measured-peak fractions
NOMINAL_HBM_GBS = 8000.0
NOMINAL_BF16_TFLOPS = 2250.0
WEIGHT_BYTES = 0.5 + 2.0 / 32  # uint4 code + BF16 scale per 32 elements
CONFIG_SET = ("tp8_16", "tp8_64", "tp8_256", "ep8_prefill", "ep8_prefill_x4",
              "grouped_contig_128", "grouped_contig_1024", "grouped_masked_32")


def make_workload(name, weights=True):
    from w4a16_int4_moe_gb300 import workloads as wl
    if name == "ep8_decode":
        return wl.ep8_decode()
    if name == "ep8_decode_e12":
        # a quarter of the EP8 decode shard (12 experts, 144 rows): the size
        # that detailed profiler captures run on
        return wl.ep8_decode(tokens=144, local_experts=12)
    if name.startswith("tp8_"):
        return wl.tp8(int(name.split("_")[1]), weights=weights)
    if name == "ep8_prefill":
        return wl.ep8_prefill(weights=weights)
    if name == "ep8_prefill_x4":
        # four times the tokens and every expert's rows (tok_e 80 .. 2400)
        return wl.ep8_prefill(weights=weights, scale=4)
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
    gu_bytes = active * i2 * h * WEIGHT_BYTES + tokens_used * h * 2 + rows * i2 * 2
    dn_bytes = active * h * i * WEIGHT_BYTES + rows * i * 2 + p.tokens * h * 4
    return {
        "gate_up": {"bytes": gu_bytes, "flops": 2.0 * rows * i2 * h},
        "down": {"bytes": dn_bytes, "flops": 2.0 * rows * h * i},
        "active_experts": active, "rows": rows,
    }


def workload_config(p, world):
    """The `config` object of both arms (identical for the same workload)."""
    flat = p.topk_ids.reshape(-1)
    local = (flat >= 0) & (flat < p.num_experts)
    return {
        "workload": p.name, "tokens": p.tokens, "hidden": p.hidden, "inter": p.inter,
        "local_experts": p.num_experts, "topk": p.topk, "routed_rows": int(local.sum()),
        "active_experts": int(np.unique(flat[local]).size),
        "l2": "flushed before every layer (256 MiB write); the weight stream exceeds L2",
        "parallelism": f"replicas x{world}",
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
    """Time the float64 oracle (as it stands) on all routed rows of
    `n_experts_sample` active experts (default: every active expert, i.e. one
    whole layer) through gate_up -> act -> down; a partial sample is scaled
    to a whole layer by the fraction of active experts sampled."""
    import oracle
    flat = p.topk_ids.reshape(-1)
    local = (flat >= 0) & (flat < p.num_experts)
    active = np.unique(flat[local])
    if n_experts_sample is None or n_experts_sample >= active.size:
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
    whole = n_experts_sample == active.size
    return {"value": dt * scale * 1e6, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
            "sample": (f"the whole layer: all {active.size} active experts" if whole else
                       f"{n_experts_sample} of {active.size} active experts, scaled x{scale:.2f}")
                      + f" (all their routed rows, {int(rows.sum())} tokens; gate_up+silu+down, "
                        f"float64 numpy), {dt:.2f} s"}


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
    vals, rec = [], None
    t0 = time.perf_counter()
    for _ in range(args.steps):
        rec = cpu_oracle_sample(p, n_experts_sample=args.ref_experts)
        vals.append(rec["value"])
    wall = time.perf_counter() - t0
    value = statistics.mean(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": wall / args.steps * 1e3, "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(p, world),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": rec["cores"],
                         "kind": "oracle", "sample": rec["sample"]},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def to_device(a, device):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def device_weights(num_experts, n, k, seed, device):
    """Seeded synthetic checkpoint tensors drawn on the device (same recipe
    as the workloads: uniform codes, |N(0,1)| * 0.02 BF16 scales)."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    q = torch.randint(0, 256, (num_experts, n, k // 2), dtype=torch.uint8, device=device,
                      generator=g)
    s = (torch.randn((num_experts, n, k // 32), device=device, generator=g).abs() * 0.02)
    return q, s.to(torch.bfloat16).view(torch.int16)


def time_indexed_layer(layer, x, tokens, ids, w, out, flush, steps, warmup, layers=1):
    """gate_up and down CUDA-event times (µs) of `steps` steps of `layers`
    layers each, L2 flushed before every layer. Returns the per-layer lists
    and the wall time of the timed steps."""
    import torch
    stream = torch.cuda.current_stream()

    def one(ev=None):
        flush.zero_()
        layer.align(ids)
        if ev is not None:
            ev[0].record(stream)
        layer.gate_up_gemm(x, tokens)
        if ev is not None:
            ev[1].record(stream)
        layer.activation(tokens)
        if ev is not None:
            ev[2].record(stream)
        layer.down_gemm(tokens, w, out)
        if ev is not None:
            ev[3].record(stream)

    for _ in range(warmup * layers):
        one()
    torch.cuda.synchronize()
    n = steps * layers
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(n)]
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(n):
        one(events[i])
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    gu = [e[0].elapsed_time(e[1]) * 1e3 for e in events]
    dn = [e[2].elapsed_time(e[3]) * 1e3 for e in events]
    return gu, dn, wall


def time_single_launch(gu_glu, dn, p, x, ids, w, out, flush, device, steps, warmup):
    """µs of the whole layer (gate_up, activation, down) in one GEMM launch
    (w4a16_moe_layer, with its row permute), L2 flushed before every step;
    None where the plan's routing blocks exceed the 128 rows the single
    launch takes."""
    import torch
    from w4a16_int4_moe_gb300 import moe as moe_mod
    from w4a16_int4_moe_gb300 import ops
    bm = ops.w4a16_plan(p.tokens, p.topk, p.num_experts, 2 * p.inter, p.hidden,
                        p.tok_e_hint()).block_m
    if bm > 128:
        return None
    layer = moe_mod.W4A16MoE(gu_glu, dn, p.topk, p.tokens, tok_e_hint=p.tok_e_hint(),
                             device=device, single_launch=True)
    stream = torch.cuda.current_stream()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    for i in range(warmup + steps):
        e = ev[i - warmup] if i >= warmup else None
        flush.zero_()
        layer.align(ids)
        if e is not None:
            e[0].record(stream)
        layer.layer_single_launch(x, p.tokens, w, out)
        if e is not None:
            e[1].record(stream)
    torch.cuda.synchronize()
    st, word = ops.w4a16_read_device_status(layer.layer_workspace)
    if st != ops.W4A16_OK:
        raise SystemExit(f"device status {word:#x} in the single-launch layer")
    return statistics.mean(e[0].elapsed_time(e[1]) * 1e3 for e in ev)


def time_e2e_pipelined(layer, host_inputs, out_shape, device, steps, warmup):
    """Per-step time of the layer through its public call with host buffers,
    pipelined as a serving loop would run it: step s's inputs are copied in
    (pinned host -> device) and its output copied back on one copy stream per
    direction, the
    layer runs on a compute stream, and two device buffer sets let the copies
    of one step overlap the compute of its neighbours. Every step still
    includes its own copies; the value is the whole run's time over steps.
    No L2 flush runs inside the pipeline (it would sit on the timed path):
    a step streams more weight bytes than L2 holds."""
    import torch
    copy_s = torch.cuda.Stream(device)    # host -> device
    back_s = torch.cuda.Stream(device)    # device -> host (the other copy direction)
    comp_s = torch.cuda.Stream(device)
    dev_in = [tuple(torch.empty(h.shape, dtype=h.dtype, device=device) for h in host_inputs)
              for _ in range(2)]
    dev_out = [torch.empty(out_shape, dtype=torch.float32, device=device) for _ in range(2)]
    host_out = [torch.empty(out_shape, dtype=torch.float32).pin_memory() for _ in range(2)]

    def run(n):
        in_ready = [torch.cuda.Event() for _ in range(n)]
        comp_done = [torch.cuda.Event() for _ in range(n)]
        out_done = [torch.cuda.Event() for _ in range(n)]
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        start.record(copy_s)
        for i in range(n + 1):
            if i < n:
                b = i % 2
                with torch.cuda.stream(copy_s):
                    if i >= 2:
                        copy_s.wait_event(comp_done[i - 2])  # buffer set b is free again
                    for d, h in zip(dev_in[b], host_inputs):
                        d.copy_(h, non_blocking=True)
                    in_ready[i].record(copy_s)
                with torch.cuda.stream(comp_s):
                    comp_s.wait_event(in_ready[i])
                    if i >= 2:
                        comp_s.wait_event(out_done[i - 2])  # its output was copied out
                    x_d, ids_d, w_d = dev_in[b]
                    layer.forward(x_d, ids_d, w_d, out=dev_out[b], stream=comp_s)
                    comp_done[i].record(comp_s)
            if i >= 1:
                j = i - 1
                with torch.cuda.stream(back_s):
                    back_s.wait_event(comp_done[j])
                    host_out[j % 2].copy_(dev_out[j % 2], non_blocking=True)
                    out_done[j].record(back_s)
        end.record(back_s)
        end.synchronize()
        return start.elapsed_time(end) * 1e3 / n

    run(warmup + 2)
    return run(steps)


def roofline_entry(bound, kernel, achieved, peak, nominal, peak_src, extra=None):
    unit = "GB/s" if bound == "hbm" else "TFLOP/s"
    d = {"bound": bound, "kernel": kernel, "achieved": achieved, "peak": peak, "unit": unit,
         "frac": achieved / peak, "peak_source": peak_src,
         "nominal_peak": nominal, "frac_of_nominal": achieved / nominal}
    if extra:
        d.update(extra)
    return d


def indexed_config(name, packed, device, flush, steps, warmup, peaks, glu_packed=None):
    """One indexed configuration (TP8 or EP8 prefill) with the given packed
    weights {(n, k): PackedExperts}: gate_up and down µs, roofline."""
    import torch
    from w4a16_int4_moe_gb300 import moe as moe_mod
    p = make_workload(name, weights=False)
    work = algorithmic_work(p)
    gu = packed[(2 * p.inter, p.hidden)]
    dn = packed[(p.hidden, p.inter)]
    layer = moe_mod.W4A16MoE(gu, dn, p.topk, p.tokens, tok_e_hint=p.tok_e_hint(), device=device)
    x = to_device(p.x.view(np.int16), device).view(torch.bfloat16)
    ids = to_device(p.topk_ids, device)
    w = to_device(p.topk_weights, device)
    out = torch.empty((p.tokens, p.hidden), dtype=torch.float32, device=device)
    gu_us, dn_us, _ = time_indexed_layer(layer, x, p.tokens, ids, w, out, flush, steps, warmup)
    torch.cuda.synchronize()
    from w4a16_int4_moe_gb300 import ops
    st, word = ops.w4a16_read_device_status(layer.workspace)
    if st != ops.W4A16_OK:
        raise SystemExit(f"device status {word:#x} in configuration {name}")
    g, d_ = statistics.mean(gu_us), statistics.mean(dn_us)
    single_us = None
    if glu_packed is not None:
        single_us = time_single_launch(glu_packed, dn, p, x, ids, w, out, flush,
                                       device, steps, warmup)
    hbm, tf, src = peaks
    tensor = name.startswith("ep8_prefill")
    layer_us = g + d_
    total_b = work["gate_up"]["bytes"] + work["down"]["bytes"]
    total_f = work["gate_up"]["flops"] + work["down"]["flops"]
    if tensor:
        roof = roofline_entry("tensor", "w4a16_moe_gemm_kernel (gate_up + down)",
                              total_f / (layer_us * 1e-6) / 1e12, tf, NOMINAL_BF16_TFLOPS,
                              f"{src} bf16_tflops")
    else:
        roof = roofline_entry("hbm", "w4a16_moe_gemm_kernel (gate_up + down)",
                              total_b / (layer_us * 1e-6) / 1e9, hbm, NOMINAL_HBM_GBS,
                              f"{src} hbm_gbs", {"algorithmic_bytes": total_b})
    return {"workload": p.name, "layer_us": layer_us, "gate_up_us": g, "down_us": d_,
            "steps": steps, "block_m": layer.block_m, "block_m_down": layer.block_m_dn,
            "routed_rows": work["rows"],
            "active_experts": work["active_experts"],
            "gate_up_gbs": work["gate_up"]["bytes"] / (g * 1e-6) / 1e9,
            "single_launch_layer_us": single_us,
            "tflops": total_f / (layer_us * 1e-6) / 1e12, "roofline": roof}


def grouped_inputs(name, device, packed):
    """(calls, label, rows, active experts) of a grouped workload on the EP8
    shard: the gate_up-shaped then the down-shaped grouped GEMM over the same
    per-expert rows, activations drawn on the device."""
    import torch
    from w4a16_int4_moe_gb300 import ops
    from w4a16_int4_moe_gb300 import workloads as wl
    g = torch.Generator(device=device)
    g.manual_seed(3)
    calls = []
    if name.startswith("grouped_contig_"):
        m = int(name.split("_")[-1])
        lay_np = wl.contiguous_layout(m, 48)
        rows = int((lay_np >= 0).sum())
        active = 48
        label = f"grouped_contiguous_E48_m{m}_H7168_I2048"
        kind = ops.W4A16_GROUPED_CONTIGUOUS
        for (n, k) in ((4096, 7168), (7168, 2048)):
            a = torch.randn((lay_np.size, k), device=device, generator=g).to(torch.bfloat16)
            out = torch.empty((lay_np.size, n), dtype=torch.bfloat16, device=device)
            calls.append((kind, packed[(n, k)], n, k, a, lay_np.size, to_device(lay_np, device),
                          m, out))
    elif name == "grouped_masked_32":
        counts = wl.masked_counts(48, 32, seed=1)
        rows = int(counts.sum())
        active = int((counts > 0).sum())
        label = "grouped_masked_E48_budget32_H7168_I2048"
        kind = ops.W4A16_GROUPED_MASKED
        for (n, k) in ((4096, 7168), (7168, 2048)):
            a = torch.randn((48, 32, k), device=device, generator=g).to(torch.bfloat16)
            out = torch.empty((48, 32, n), dtype=torch.bfloat16, device=device)
            calls.append((kind, packed[(n, k)], n, k, a, 32, to_device(counts, device), 16, out))
    else:
        raise SystemExit(f"unknown workload {name}")
    return calls, label, rows, active


def grouped_work(rows, active):
    """Algorithmic bytes and flops of one grouped step on the EP8 shard: the
    weights of the experts with rows, each valid BF16 input row read once and
    each valid BF16 output row written once, 2 * rows * n * k flops per GEMM."""
    gu_bytes = active * 4096 * 7168 * WEIGHT_BYTES + rows * 7168 * 2 + rows * 4096 * 2
    dn_bytes = active * 7168 * 2048 * WEIGHT_BYTES + rows * 2048 * 2 + rows * 7168 * 2
    return {"gate_up": {"bytes": gu_bytes, "flops": 2.0 * rows * 4096 * 7168},
            "down": {"bytes": dn_bytes, "flops": 2.0 * rows * 7168 * 2048}}


def grouped_config(name, packed, device, flush, steps, warmup, peaks):
    """One step = the grouped gate_up GEMM then the grouped down GEMM (the
    activation between them untimed), L2 flushed before each step."""
    import torch
    from w4a16_int4_moe_gb300 import ops
    calls, label, rows, active = grouped_inputs(name, device, packed)
    ws = torch.zeros(256, dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream()

    def run(c):
        kind, pk, n, k, a, m, lay, exp_m, out = c
        ops.w4a16_moe_grouped_gemm(kind, pk.packed, 48, n, k, a, m, lay, ws, expected_m=exp_m,
                                   out=out)

    for _ in range(warmup):
        flush.zero_()
        run(calls[0])
        run(calls[1])
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(steps):
        flush.zero_()
        ev[i][0].record(stream)
        run(calls[0])
        ev[i][1].record(stream)
        run(calls[1])
        ev[i][2].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    st, word = ops.w4a16_read_device_status(ws)
    if st != ops.W4A16_OK:
        raise SystemExit(f"device status {word:#x} in configuration {name}")
    gu_us = statistics.mean(e[0].elapsed_time(e[1]) * 1e3 for e in ev)
    dn_us = statistics.mean(e[1].elapsed_time(e[2]) * 1e3 for e in ev)
    work = grouped_work(rows, active)
    gu_bytes, dn_bytes = work["gate_up"]["bytes"], work["down"]["bytes"]
    flops = work["gate_up"]["flops"] + work["down"]["flops"]
    layer_us = gu_us + dn_us
    hbm, tf, src = peaks
    if name.startswith("grouped_contig_"):
        roof = roofline_entry("tensor", "w4a16_moe_gemm_kernel (grouped gate_up + down)",
                              flops / (layer_us * 1e-6) / 1e12, tf, NOMINAL_BF16_TFLOPS,
                              f"{src} bf16_tflops")
    else:
        roof = roofline_entry("hbm", "w4a16_moe_gemm_kernel (grouped gate_up + down)",
                              (gu_bytes + dn_bytes) / (layer_us * 1e-6) / 1e9, hbm,
                              NOMINAL_HBM_GBS, f"{src} hbm_gbs",
                              {"algorithmic_bytes": gu_bytes + dn_bytes})
    return {"workload": label, "layer_us": layer_us, "gate_up_us": gu_us, "down_us": dn_us,
            "steps": steps, "valid_rows": rows, "tflops": flops / (layer_us * 1e-6) / 1e12,
            "wall_s": wall, "roofline": roof}


def run_configs(args, packed_ep8, device, flush, peaks):
    """The `configs` block: every other configuration, measured in this run."""
    import torch
    from w4a16_int4_moe_gb300 import moe as moe_mod
    from w4a16_int4_moe_gb300 import ops
    steps = max(3, min(args.steps, 20))
    warmup = max(3, min(args.warmup, 5))
    res = {}
    packed = dict(packed_ep8)
    tp8_packed = None
    for name in CONFIG_SET:
        t0 = time.perf_counter()
        if name.startswith("tp8_"):
            if tp8_packed is None:
                q, s = device_weights(384, 512, 7168, 11, device)
                gu = moe_mod.PackedExperts.from_checkpoint(q, s)
                tp8_glu = moe_mod.PackedExperts.from_checkpoint(
                    q, s, layout=ops.W4A16_LAYOUT_KTILE64_GLU16)
                del q, s
                q, s = device_weights(384, 7168, 256, 12, device)
                dn = moe_mod.PackedExperts.from_checkpoint(q, s)
                del q, s
                tp8_packed = {(512, 7168): gu, (7168, 256): dn}
            r = indexed_config(name, tp8_packed, device, flush, steps, warmup, peaks,
                               glu_packed=tp8_glu)
        elif name.startswith("ep8_prefill"):
            r = indexed_config(name, packed, device, flush, steps, warmup, peaks)
        else:
            r = grouped_config(name, packed, device, flush, steps, warmup, peaks)
        r["setup_and_run_s"] = time.perf_counter() - t0
        res[name] = r
        torch.cuda.empty_cache()
    return res


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

    gu = moe_mod.PackedExperts.from_checkpoint(to_device(p.q_gu, device),
                                               to_device(p.s_gu.view(np.int16), device))
    dn = moe_mod.PackedExperts.from_checkpoint(to_device(p.q_dn, device),
                                               to_device(p.s_dn.view(np.int16), device))
    layer = moe_mod.W4A16MoE(gu, dn, p.topk, p.tokens, tok_e_hint=p.tok_e_hint(), device=device)
    x = to_device(p.x.view(np.int16), device).view(torch.bfloat16)
    ids = to_device(p.topk_ids, device)
    w = to_device(p.topk_weights, device)
    out = torch.empty((p.tokens, p.hidden), dtype=torch.float32, device=device)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream()
    L = max(1, args.layers)

    clocks = ClockSampler()
    clocks.start()
    if dist is not None:
        dist.barrier()
    gu_us, dn_us, wall = time_indexed_layer(layer, x, p.tokens, ids, w, out, flush, args.steps,
                                            args.warmup, layers=L)
    t_end_wall = time.time()
    clocks.mark(t_end_wall - wall, t_end_wall)
    if dist is not None:
        dist.barrier()
    clk = clocks.stop()
    st, word = ops.w4a16_read_device_status(layer.workspace)
    if st != ops.W4A16_OK:
        raise SystemExit(f"device status {word:#x} after the timed steps")
    layer_us = statistics.mean(a + b for a, b in zip(gu_us, dn_us))
    layer_us = reduce_max(layer_us, dist)
    wall = reduce_max(wall, dist)
    value = layer_us / world   # replicas: world layers per layer time

    # ---- the layer with the activation fused into gate_up (reported
    # beside the metric; the metric itself keeps the activation untimed) ----
    fused = None
    layer_f = None
    if not args.no_fused:
        gu_glu = moe_mod.PackedExperts.from_checkpoint(
            to_device(p.q_gu, device), to_device(p.s_gu.view(np.int16), device),
            layout=ops.W4A16_LAYOUT_KTILE64_GLU16)
        layer_f = moe_mod.W4A16MoE(gu_glu, dn, p.topk, p.tokens, tok_e_hint=p.tok_e_hint(),
                                   device=device)
        nf = max(20, args.steps)
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
        single_us = time_single_launch(gu_glu, dn, p, x, ids, w, out, flush, device, nf,
                                       args.warmup)
        fused = {
            "gate_up_silu_us": statistics.mean(e[0].elapsed_time(e[1]) * 1e3 for e in ev_f),
            "down_us": statistics.mean(e[1].elapsed_time(e[2]) * 1e3 for e in ev_f),
            "layer_with_act_us": statistics.mean(e[0].elapsed_time(e[2]) * 1e3 for e in ev_f),
            "unfused_layer_with_act_us": statistics.mean(e[3].elapsed_time(e[4]) * 1e3
                                                         for e in ev_f),
            "single_launch_layer_us": single_us,
            "steps": nf,
        }

    # ---- end to end through the public call, host buffers: the layer a user
    # builds, with the activation fused into gate_up when measured above ----
    e2e_layer = layer_f if layer_f is not None else layer
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
    for _ in range(max(20, args.steps)):
        flush.zero_()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        e2e_step()
        e1.record(stream)
        e1.synchronize()
        e2e_times.append(e0.elapsed_time(e1) * 1e3)
    e2e_serial_us = reduce_max(statistics.mean(e2e_times), dist) / world
    e2e_us = reduce_max(time_e2e_pipelined(e2e_layer, (x_h, ids_h, w_h), out_h.shape,
                                           device, max(20, args.steps), max(1, args.warmup)),
                        dist) / world
    h2d = p.x.nbytes + p.topk_ids.nbytes + p.topk_weights.nbytes
    d2h = p.tokens * p.hidden * 4

    peaks = measured_peaks()
    configs = None
    if not args.no_configs and rank == 0 and args.workload == "ep8_decode":
        configs = run_configs(args, {(2 * p.inter, p.hidden): gu, (p.hidden, p.inter): dn},
                              device, flush, peaks)

    if rank != 0:
        return
    hbm, tflops_peak, peak_src = peaks
    gu_mean = statistics.mean(gu_us)
    dn_mean = statistics.mean(dn_us)
    gu_gbs = work["gate_up"]["bytes"] / (gu_mean * 1e-6) / 1e9
    dn_gbs = work["down"]["bytes"] / (dn_mean * 1e-6) / 1e9
    total_bytes = work["gate_up"]["bytes"] + work["down"]["bytes"]
    total_flops = work["gate_up"]["flops"] + work["down"]["flops"]
    layer_gbs = total_bytes / (layer_us * 1e-6) / 1e9
    traffic = traffic_record(os.path.join(ROOT, "w4a16_int4_moe_gb300", "csrc", "moe_gemm.cu"),
                             args.workload)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": wall / args.steps * 1e3,
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded; random uint4 weights, N(0,1) activations)",
        "config": workload_config(p, world),
        "layers_per_step": L,
        "plan": {"block_m": layer.block_m, "gate_up": layer.plan_gu.as_dict(),
                 "down": layer.plan_dn.as_dict()},
        "gate_up_us": gu_mean, "down_us": dn_mean,
        "achieved": {"hbm_gbs": layer_gbs, "tflops": total_flops / (layer_us * 1e-6) / 1e12,
                     "gate_up_gbs": gu_gbs, "down_gbs": dn_gbs},
        "roofline": roofline_entry(
            "hbm", "w4a16_moe_gemm_kernel (gate_up)", gu_gbs, hbm, NOMINAL_HBM_GBS,
            f"{peak_src} hbm_gbs",
            {"traffic": None if traffic is None else traffic["dram_bytes_per_launch"],
             "algorithmic_bytes": work["gate_up"]["bytes"]}),
        "layer_roofline": roofline_entry(
            "hbm", "w4a16_moe_gemm_kernel (gate_up + down)", layer_gbs, hbm, NOMINAL_HBM_GBS,
            f"{peak_src} hbm_gbs", {"algorithmic_bytes": total_bytes}),
        # the same bytes over the single-launch layer (gate_up with the fused
        # activation, then down, one launch), when measured
        "single_launch_roofline": (roofline_entry(
            "hbm", "w4a16_moe_gemm_kernel (single-launch layer)",
            total_bytes / (fused["single_launch_layer_us"] * 1e-6) / 1e9, hbm, NOMINAL_HBM_GBS,
            f"{peak_src} hbm_gbs", {"layer_us": fused["single_launch_layer_us"],
                                    "algorithmic_bytes": total_bytes})
            if fused and fused.get("single_launch_layer_us") else None),
        # per layer: align, permute + gate_up, silu, permute + down
        "gpu_launches": 6 * L * args.steps,
        "e2e": {"value": e2e_us, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "serial_value": e2e_serial_us,
                "pipeline": ("every step copies its inputs in from pinned host memory and its "
                             "output back, one copy stream per direction; the layer runs on a "
                             "compute stream; "
                             "two device buffer sets let step s's copies overlap the compute of "
                             "steps s-1 and s+1; no L2 flush between steps (a step streams more "
                             "weight bytes than L2 holds). serial_value: one step at a time on "
                             "one stream, L2 flushed before each step outside the timed region"),
                "call": ("W4A16MoE.forward (align, then gate_up with the fused activation and "
                         "down in one launch)" if layer_f is not None and layer_f.single_launch
                         else "W4A16MoE.forward (align, gate_up with fused activation, down)"
                         if layer_f is not None
                         else "W4A16MoE.forward (align, gate_up, act, down)")},
        "clocks": clk,
        "fused_activation": fused,
        "configs": configs,
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_oracle_sample(p)
    print(json.dumps(line))


def run_grouped(args):
    """A grouped workload as the headline (weights drawn on the device)."""
    import torch
    from w4a16_int4_moe_gb300 import moe as moe_mod
    from w4a16_int4_moe_gb300 import ops
    torch.cuda.set_device(0)
    device = torch.device("cuda", 0)
    ops.load_library()
    packed = {}
    for (n, k), seed in (((4096, 7168), 1), ((7168, 2048), 2)):
        q, s = device_weights(48, n, k, seed, device)
        packed[(n, k)] = moe_mod.PackedExperts.from_checkpoint(q, s)
        del q, s
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    clocks = ClockSampler()
    clocks.start()
    r = grouped_config(args.workload, packed, device, flush, args.steps, args.warmup,
                       measured_peaks())
    t_end = time.time()
    clocks.mark(t_end - r["wall_s"], t_end)
    clk = clocks.stop()
    line = {
        "metric": METRIC, "value": r["layer_us"], "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": r["wall_s"] / args.steps * 1e3, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded; random uint4 weights, N(0,1) activations)",
        "config": {"workload": r["workload"], "valid_rows": r["valid_rows"], "experts": 48,
                   "l2": "flushed before every step (256 MiB write)"},
        "gate_up_us": r["gate_up_us"], "down_us": r["down_us"], "tflops": r["tflops"],
        "roofline": r["roofline"], "gpu_launches": 2 * args.steps, "clocks": clk,
    }
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--layers", type=int, default=32,
                    help="MoE layers per step (each streams the weights after an L2 flush)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="ep8_decode")
    ap.add_argument("--ref-experts", type=int, default=None,
                    help="reference arm: experts per step (default: every active expert, "
                         "the whole layer)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-fused", action="store_true",
                    help="skip the fused-activation layer measurement")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the other configurations (the `configs` object)")
    args = ap.parse_args()
    if args.impl == "reference":
        run_reference(args)
    elif args.workload.startswith("grouped_"):
        run_grouped(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
