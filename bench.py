"""Benchmark of the CRISP sparse-prefill path on one GB300 (one JSON line on stdout).

A step is one full pass of the path over one attention layer of synthetic input:
crisp_select (PatSearch proxy, C_struct routing, VS / PE selection, CSR build) followed
by crisp_attend (block-sparse exact attention), i.e. crisp_prefill.  The default
workload is the Llama-3-8B layer shape at 512k tokens (32 query heads, 8 KV heads,
d = 128, planted VS/PE mix, alpha = 1.0); inputs (4.3 GB of Q) exceed the 129 MB L2, so
no flush is needed between steps.

Reported: ms per layer (value), effective TFLOP/s over the selected blocks, per-phase
times, the speedup over the in-library dense causal kernel on the same inputs, the
attention kernel's roofline fraction, an end-to-end number with host buffers, and the
CPU oracle timed on a bounded sample of the same workload.

--impl reference times the CPU oracle alone (the reference arm of this build).
Multi-GPU: the path is run as independent replicas (one layer per rank, no collective).
"""
import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = ("sparse prefill attn ms/layer and TFLOP/s at 128k/512k; speedup vs in-build dense")
UNIT = "ms/layer"
B = 128
D = 128
def launches_per_prefill(w, sms: int) -> int:
    """Kernel launches of one crisp_prefill, as the library plans them (selection, work
    order, the fast attention kernel once per group of KV heads, the rescue pass)."""
    import dynamic_sparse_prefill_gb300 as dsp
    return dsp.prefill_launches(dsp.make_dims(w.batch, w.n, w.hq, w.hkv), sms)


def algorithmic_flops(nnz: int, rows: int) -> float:
    """4*B^2*d per off-diagonal block pair (QK^T and PV), 2*d*B*(B+1) per causal diagonal."""
    return 4.0 * B * B * D * (nnz - rows) + 2.0 * D * B * (B + 1) * rows


def kernel_code_hash(path: str) -> str:
    """sha256 of a CUDA source with // comments and blank lines removed: the counters of a
    capture stay valid while only the comments change."""
    import hashlib
    import re
    lines = []
    for line in open(path).read().splitlines():
        line = re.sub(r"//.*$", "", line).rstrip()
        if line.strip():
            lines.append(line)
    return hashlib.sha256("\n".join(lines).encode()).hexdigest()


def recorded_traffic(workload: str):
    """DRAM bytes of one crisp_attend (summed over its attention-kernel launches) from the
    committed ncu summary, if it was taken on this workload with the current kernel code;
    else None."""
    import re
    prof = os.path.join(ROOT, "profiles", f"attention_kernel_{workload}_traffic.md")
    src = os.path.join(ROOT, "dynamic_sparse_prefill_gb300", "csrc", "attention.cu")
    if not os.path.exists(prof):
        return None
    text = open(prof).read()
    m = re.search(r"code_sha256: ([0-9a-f]{64})", text)
    rd = re.search(r"dram_bytes_read: (\d+)", text)
    wr = re.search(r"dram_bytes_write: (\d+)", text)
    if not (m and rd and wr):
        return None
    if kernel_code_hash(src) != m.group(1):
        return None
    return int(rd.group(1)) + int(wr.group(1))


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return j, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.rows = []
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(self.dev)], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append([x.strip() for x in line.split(",")])

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        sm = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in self.rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in self.rows:
            for i, nm in enumerate(names):
                if len(r) > 5 + i and r[5 + i].lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(self.rows)}


def make_inputs(w):
    from workloads.planted import generate
    return generate(w)


def cpu_oracle_sample(w, g, stats, budget_s=20.0):
    """Times the fp64 CPU oracle on a bounded sample of the workload and extrapolates to
    one layer: full selection of one VS-planted and one PE-planted head, and the exact
    attention of a few query blocks (per selected block pair)."""
    from oracle import crisp_oracle as O
    params = O.workload_params(w)
    pe_set = set(w.pe_heads)
    vs_h = next(h for h in range(w.hq) if h not in pe_set)
    pe_h = next((h for h in range(w.hq) if h in pe_set), None)
    t_sel = {}
    sels = {}
    for h in [vs_h] + ([pe_h] if pe_h is not None else []):
        q = O.bf16_bits_to_f64(g["q"][h])
        k = O.bf16_bits_to_f64(g["k"][h // w.group])
        t0 = time.perf_counter()
        sels[h] = O.crisp_select_head(q, k, **params)
        t_sel[h] = time.perf_counter() - t0
    # attention: sampled query blocks of the PE head (long rows) until ~budget/2 seconds
    h = pe_h if pe_h is not None else vs_h
    q = O.bf16_bits_to_f64(g["q"][h])
    k = O.bf16_bits_to_f64(g["k"][h // w.group])
    v = O.bf16_bits_to_f64(g["v"][h // w.group])
    mask = sels[h]["mask"]
    rng = np.random.default_rng(5)
    nb = w.n_blocks
    pairs, t_att, blocks = 0, 0.0, 0
    t_start = time.perf_counter()
    while time.perf_counter() - t_start < budget_s / 2 and blocks < nb:
        I = int(rng.integers(nb // 2, nb))
        t0 = time.perf_counter()
        O.block_sparse_attention(q, k, v, mask, w.B, [I])
        t_att += time.perf_counter() - t0
        pairs += int(mask[I, : I + 1].sum())
        blocks += 1
    per_pair = t_att / max(pairs, 1)
    n_pe = stats["n_pe"]
    n_vs = stats["n_vs"]
    sel_s = t_sel[vs_h] * n_vs + (t_sel[pe_h] if pe_h is not None else t_sel[vs_h]) * n_pe
    total_s = sel_s + per_pair * stats["nnz"]
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    sample = (f"oracle selection of head {vs_h} (VS) and head {pe_h} (PE) in full "
              f"({t_sel[vs_h]:.2f} s, {t_sel.get(pe_h, 0):.2f} s); exact attention of "
              f"{blocks} query blocks ({pairs} block pairs, {t_att:.2f} s); extrapolated "
              f"to {n_vs} VS + {n_pe} PE heads and {stats['nnz']} block pairs")
    return {"value": total_s * 1e3, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": sample, "extrapolated": True,
            "measured_s": sum(t_sel.values()) + t_att}


def run_reference(args, w, rank, world):
    """The reference arm: the CPU oracle as it stands, on bounded samples."""
    if rank != 0:
        return
    g = make_inputs(w)
    # expected selection sizes from the oracle itself (full selection is part of the sample)
    from oracle import crisp_oracle as O
    params = O.workload_params(w)
    pe_set = set(w.pe_heads)
    n_pe = sum(1 for h in range(w.hq) if h in pe_set)
    vals = []
    for step in range(args.warmup + args.steps):
        # per step: the selection of one VS and one PE head, plus sampled attention rows;
        # the layer's pair count is estimated from those two heads' masks.
        vs_h = next(h for h in range(w.hq) if h not in pe_set)
        pe_h = next((h for h in range(w.hq) if h in pe_set), vs_h)
        nnz = 0
        for h, mult in ((vs_h, w.hq - n_pe), (pe_h, n_pe)):
            q = O.bf16_bits_to_f64(g["q"][h])
            k = O.bf16_bits_to_f64(g["k"][h // w.group])
            r = O.crisp_select_head(q, k, **params)
            nnz += int(np.tril(r["mask"]).sum()) * mult
        stats = {"n_vs": w.hq - n_pe, "n_pe": n_pe, "nnz": nnz}
        cb = cpu_oracle_sample(w, g, stats, budget_s=args.ref_budget)
        if step >= args.warmup:
            vals.append(cb["value"])
    value = statistics.mean(vals)
    cb["value"] = value
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": value, "higher_is_better": False, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (planted, seeded)",
            "config": workload_config(w), "cpu_baseline": cb,
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def workload_config(w):
    return {"workload": w.name, "n": w.n, "hq": w.hq, "hkv": w.hkv, "d": w.d, "batch": w.batch,
            "alpha": w.alpha, "gamma": w.gamma, "tau_proxy": w.tau_proxy, "B": w.B,
            "k_min_tokens": w.k_min_tokens, "l2": l2_note(w)}


L2_BYTES = 129e6


def l2_note(w) -> str:
    q_bytes = w.batch * w.hq * w.n * w.d * 2
    if q_bytes > L2_BYTES:
        return "inputs larger than L2 (Q alone is %.2f GB); no flush" % (q_bytes / 1e9)
    return "inputs smaller than L2 (Q is %.1f MB): timings include L2 reuse" % (q_bytes / 1e6)


def max_over_ranks(value: float) -> float:
    """Max of a per-rank number over all ranks (the slowest replica sets the step time)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    dev = torch.device("cuda", torch.cuda.current_device()) \
        if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_value(ms_per_step: float, world: int) -> float:
    """ms per layer of the whole job: `world` replicas each process one layer per step."""
    return ms_per_step / world


def run_gpu(args, w, rank, world):
    import torch
    import torch.distributed as dist
    import dynamic_sparse_prefill_gb300 as dsp

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    g = make_inputs(w)

    def dev_tensor(u16):
        return torch.from_numpy(u16.view(np.int16)).view(torch.bfloat16).to(dev)

    q, k, v = dev_tensor(g["q"]), dev_tensor(g["k"]), dev_tensor(g["v"])
    o = torch.empty_like(q)
    dims = dsp.make_dims(1, w.n, w.hq, w.hkv)
    ctx = dsp.Context(dims)
    flags = {"none": 0, "median": dsp.FLAG_MEDIAN_FLOOR,
             "gamma": dsp.FLAG_VS_GAMMA_CUMSUM}[args.vs_variant]
    cfg = dsp.default_cfg(alpha=w.alpha, gamma=w.gamma, tau_proxy=w.tau_proxy,
                          k_min_tokens=w.k_min_tokens, flags=flags)
    stream = torch.cuda.current_stream()

    for _ in range(args.warmup):
        ctx.prefill(dims, q, k, v, cfg, o)
    if ctx.sync_status() != 0:
        raise RuntimeError("device error during warm-up")
    stats = ctx.stats(dims)

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(dev.index) as clk:
        t_start.record(stream)
        for i in range(args.steps):
            ev[i][0].record(stream)
            ctx.select(dims, q, k, cfg)
            ev[i][1].record(stream)
            ctx.attend(dims, q, k, v, o)
            ev[i][2].record(stream)
        t_end.record(stream)
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    if ctx.sync_status() != 0:
        raise RuntimeError("device error during the timed region")
    total_ms = max_over_ranks(t_start.elapsed_time(t_end))
    sel_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
    att_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in ev)
    ms_per_step = total_ms / args.steps
    value = replica_value(ms_per_step, world)

    # end to end through the public API with host buffers (pinned), copies included:
    # crisp_prefill_host uploads, computes and downloads chunk by chunk, overlapped
    qh = torch.from_numpy(g["q"].view(np.int16)).view(torch.bfloat16).pin_memory()
    kh = torch.from_numpy(g["k"].view(np.int16)).view(torch.bfloat16).pin_memory()
    vh = torch.from_numpy(g["v"].view(np.int16)).view(torch.bfloat16).pin_memory()
    oh = torch.empty(o.shape, dtype=torch.bfloat16).pin_memory()
    e2e_steps = max(1, min(args.steps, 3))
    ctx.prefill_host(dims, qh, kh, vh, cfg, oh, q, k, v, o)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        ctx.prefill_host(dims, qh, kh, vh, cfg, oh, q, k, v, o)
    e1.record(stream)
    torch.cuda.synchronize()
    if ctx.sync_status() != 0:
        raise RuntimeError("device error in the end-to-end run")
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    h2d = int(qh.numel() + kh.numel() + vh.numel()) * 2
    d2h = int(oh.numel()) * 2

    # dense causal attention on the same inputs (the speedup denominator)
    dense_ms = None
    if not args.no_dense:
        ctx.dense(dims, q, k, v, o)
        torch.cuda.synchronize()
        de = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        de[0].record(stream)
        for _ in range(args.dense_steps):
            ctx.dense(dims, q, k, v, o)
        de[1].record(stream)
        torch.cuda.synchronize()
        dense_ms = de[0].elapsed_time(de[1]) / args.dense_steps
        if ctx.sync_status() != 0:
            raise RuntimeError("device error in dense attention")

    if rank != 0:
        return
    peaks, peak_kind = load_peaks()
    flops = algorithmic_flops(stats["nnz"], stats["rows"])
    att_tflops = flops / (att_ms * 1e-3) / 1e12
    peak = float(peaks.get("bf16_tflops_sustained", peaks.get("bf16_tflops")))
    nbk = w.n // B
    dense_flops = algorithmic_flops(w.hq * nbk * (nbk + 1) // 2, w.hq * nbk)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (planted, seeded); no real-model activations",
        "config": dict(workload_config(w), vs_variant=args.vs_variant),
        "tflops_effective": flops / (ms_per_step * 1e-3) / 1e12,
        "select_ms": sel_ms, "attend_ms": att_ms, "attend_tflops": att_tflops,
        "dense_ms": dense_ms,
        "dense_tflops": (dense_flops / (dense_ms * 1e-3) / 1e12) if dense_ms else None,
        "speedup_vs_dense": (dense_ms / ms_per_step) if dense_ms else None,
        "selection": {"nnz_block_pairs": stats["nnz"], "rows": stats["rows"],
                      "density": stats["nnz"] / (w.hq * nbk * (nbk + 1) / 2),
                      "n_vs": stats["n_vs"], "n_pe": stats["n_pe"],
                      "pe_rescued_rows": stats["pe_rescued"], "max_row": stats["max_row"]},
        "roofline": {"kernel": "attention_kernel", "bound": "tensor", "achieved": att_tflops,
                     "peak": peak, "unit": "TFLOP/s", "frac": att_tflops / peak,
                     "peak_kind": f"bf16 sustained, {peak_kind}",
                     "traffic": recorded_traffic(w.name),
                     "unit_of_work": "one crisp_attend call (all launches of the attention "
                                     "kernels for the layer)",
                     "algorithmic_flops_per_attend": flops},
        "gpu_launches": launches_per_prefill(w, torch.cuda.get_device_properties(0).multi_processor_count) * args.steps,
        "e2e": {"value": e2e_ms / world, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "clocks": clk.summary(),
        "pages_context": {"crisp_speedup_vs_flashattention_512k_h100": 5.30},
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_oracle_sample(w, g, stats, budget_s=args.ref_budget)
    print(json.dumps(line), flush=True)
    ctx.close()


def run_sweep(args):
    """Latency over sequence length (Llama-3-8B layer shape, 8k .. 512k): crisp_prefill and
    crisp_dense per layer on the same seeded inputs, one JSON line per length, then the
    estimated sparse/dense crossover length (log-log interpolation of the speedup)."""
    import torch
    import dynamic_sparse_prefill_gb300 as dsp
    from workloads import get
    from workloads.configs import SWEEP
    torch.cuda.set_device(0)
    stream = torch.cuda.current_stream()
    pts, pts_g = [], []
    for name in SWEEP:
        w = get(name)
        g = make_inputs(w)
        dev_t = lambda u16: torch.from_numpy(u16.view(np.int16)).view(torch.bfloat16).cuda()
        q, k, v = dev_t(g["q"]), dev_t(g["k"]), dev_t(g["v"])
        del g
        o = torch.empty_like(q)
        dims = dsp.make_dims(1, w.n, w.hq, w.hkv)
        ctx = dsp.Context(dims)
        cfg = dsp.default_cfg(alpha=w.alpha, gamma=w.gamma, tau_proxy=w.tau_proxy,
                              k_min_tokens=w.k_min_tokens)

        def timed(fn, reps):
            fn()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(reps):
                fn()
            e1.record(stream)
            torch.cuda.synchronize()
            return e0.elapsed_time(e1) / reps

        reps = 10 if w.n <= 65536 else 3
        sel_ms = timed(lambda: ctx.select(dims, q, k, cfg), reps)
        pre_ms = timed(lambda: ctx.prefill(dims, q, k, v, cfg, o), reps)
        # the same call replayed from a captured CUDA graph (the first call captures it)
        gcfg = dsp.default_cfg(alpha=w.alpha, gamma=w.gamma, tau_proxy=w.tau_proxy,
                               k_min_tokens=w.k_min_tokens, flags=dsp.FLAG_GRAPH_REPLAY)
        pre_g_ms = timed(lambda: ctx.prefill(dims, q, k, v, gcfg, o), reps)
        att_ms = timed(lambda: ctx.attend(dims, q, k, v, o), reps)
        den_ms = timed(lambda: ctx.dense(dims, q, k, v, o), max(1, reps // 2))
        if ctx.sync_status() != 0:
            raise RuntimeError(f"device error in the sweep at {name}")
        st = ctx.stats(dims)
        nbk = w.n // B
        line = {"sweep": True, "workload": name, "n": w.n, "prefill_ms": pre_ms,
                "prefill_graph_ms": pre_g_ms,
                "select_ms": sel_ms, "attend_ms": att_ms, "dense_ms": den_ms,
                "speedup_vs_dense": den_ms / pre_ms,
                "speedup_vs_dense_graph": den_ms / pre_g_ms,
                "attend_tflops": algorithmic_flops(st["nnz"], st["rows"]) / (att_ms * 1e-3) / 1e12,
                "dense_tflops": algorithmic_flops(w.hq * nbk * (nbk + 1) // 2, w.hq * nbk)
                / (den_ms * 1e-3) / 1e12,
                "density": st["nnz"] / (w.hq * nbk * (nbk + 1) / 2)}
        print(json.dumps(line), flush=True)
        pts.append((w.n, den_ms / pre_ms))
        pts_g.append((w.n, den_ms / pre_g_ms))
        ctx.close()
        del q, k, v, o
        torch.cuda.empty_cache()
    def crossover(p):
        for (n0, s0), (n1, s1) in zip(p, p[1:]):
            if s0 < 1.0 <= s1:
                f = (math.log(1.0) - math.log(s0)) / (math.log(s1) - math.log(s0))
                return math.exp(math.log(n0) + f * (math.log(n1) - math.log(n0)))
        if p and p[0][1] >= 1.0:
            return f"below {p[0][0]}"
        return None

    print(json.dumps({"sweep_summary": True, "crossover_tokens": crossover(pts),
                      "crossover_tokens_graph": crossover(pts_g),
                      "speedups": {n: s for n, s in pts},
                      "speedups_graph": {n: s for n, s in pts_g}}), flush=True)


def run_jsd(args):
    """Routing-signal comparison: FlexPrefill's JSD (crisp_jsd) against C_struct on the
    same heads -- cost of the extra pooled estimate and KL passes, and agreement of the
    two routes.  One JSON line per workload."""
    import torch
    import dynamic_sparse_prefill_gb300 as dsp
    from workloads import get
    torch.cuda.set_device(0)
    stream = torch.cuda.current_stream()
    for name in ("llama8b_n32k", "llama8b_n128k_a1", "qwen7b_n128k", "llama8b_n512k"):
        w = get(name)
        g = make_inputs(w)
        dev_t = lambda u16: torch.from_numpy(u16.view(np.int16)).view(torch.bfloat16).cuda()
        q, k = dev_t(g["q"]), dev_t(g["k"])
        del g
        dims = dsp.make_dims(1, w.n, w.hq, w.hkv)
        ctx = dsp.Context(dims)
        cfg = dsp.default_cfg(alpha=w.alpha, gamma=w.gamma, tau_proxy=w.tau_proxy)
        d_js = torch.zeros(w.hq, dtype=torch.float32, device="cuda")
        rt = torch.zeros(w.hq, dtype=torch.uint8, device="cuda")
        ctx.select(dims, q, k, cfg)
        ctx.jsd(dims, q, k, args.tau_jsd, d_js, rt)
        torch.cuda.synchronize()
        e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        reps = 5
        e[0].record(stream)
        for _ in range(reps):
            ctx.select(dims, q, k, cfg)
        e[1].record(stream)
        for _ in range(reps):
            ctx.jsd(dims, q, k, args.tau_jsd, d_js, rt)
        e[2].record(stream)
        torch.cuda.synchronize()
        if ctx.sync_status() != 0:
            raise RuntimeError("device error in the JSD comparison")
        sel = ctx.selection_get(dims, with_csr=False)
        routes = rt.cpu().numpy()
        agree = int((routes == sel["route_vs"]).sum())
        print(json.dumps({"jsd": True, "workload": name, "n": w.n, "tau_jsd": args.tau_jsd,
                          "select_ms": e[0].elapsed_time(e[1]) / reps,
                          "jsd_extra_ms": e[1].elapsed_time(e[2]) / reps,
                          "route_agreement": agree / w.hq,
                          "d_js": [round(float(x), 5) for x in d_js.cpu().numpy()]}), flush=True)
        ctx.close()
        del q, k
        torch.cuda.empty_cache()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="crisp", choices=["crisp", "reference"])
    ap.add_argument("--workload", default="llama8b_n512k")
    ap.add_argument("--dense-steps", type=int, default=2)
    ap.add_argument("--no-dense", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ref-budget", type=float, default=12.0)
    ap.add_argument("--vs-variant", default="none", choices=["none", "median", "gamma"],
                    help="VS selection variant: median noise floor, or FlexPrefill's "
                         "gamma-cumsum budget (the Abl.1 rule)")
    ap.add_argument("--jsd", action="store_true",
                    help="JSD vs C_struct routing comparison (one line per workload)")
    ap.add_argument("--tau-jsd", type=float, default=0.1)
    ap.add_argument("--sweep", action="store_true",
                    help="latency sweep 8k..512k (one line per length), not the bench line")
    args = ap.parse_args()
    if args.sweep:
        run_sweep(args)
        return
    if args.jsd:
        run_jsd(args)
        return
    from workloads import get
    w = get(args.workload)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        run_reference(args, w, rank, world)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        dist.init_process_group("nccl")
    run_gpu(args, w, rank, world)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
