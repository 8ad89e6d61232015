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
    one layer: the full selection of one VS-planted and one PE-planted head, and the exact
    attention of sampled query blocks of both heads, timed per selected block pair
    separately for VS rows (a few tens of scattered blocks) and PE rows (long runs), then
    weighted by the layer's VS and PE pair counts (stats: n_vs, n_pe, nnz_vs, nnz_pe)."""
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
    rng = np.random.default_rng(5)
    nb = w.n_blocks
    per_pair, desc, t_att_total = {}, [], 0.0
    heads = [("vs", vs_h)] + ([("pe", pe_h)] if pe_h is not None else [])
    for kind, h in heads:
        q = O.bf16_bits_to_f64(g["q"][h])
        k = O.bf16_bits_to_f64(g["k"][h // w.group])
        v = O.bf16_bits_to_f64(g["v"][h // w.group])
        mask = sels[h]["mask"]
        pairs, t_att, blocks = 0, 0.0, 0
        t_start = time.perf_counter()
        while time.perf_counter() - t_start < budget_s / (2 * len(heads)) and blocks < nb:
            I = int(rng.integers(nb // 2, nb))
            t0 = time.perf_counter()
            O.block_sparse_attention(q, k, v, mask, w.B, [I])
            t_att += time.perf_counter() - t0
            pairs += int(mask[I, : I + 1].sum())
            blocks += 1
        per_pair[kind] = t_att / max(pairs, 1)
        t_att_total += t_att
        desc.append(f"exact attention of {blocks} query blocks of head {h} ({kind.upper()}, "
                    f"{pairs} block pairs, {t_att:.2f} s)")
    n_pe, n_vs = stats["n_pe"], stats["n_vs"]
    nnz_vs = stats.get("nnz_vs", stats["nnz"] if pe_h is None else 0)
    nnz_pe = stats.get("nnz_pe", stats["nnz"] - nnz_vs)
    sel_s = t_sel[vs_h] * n_vs + (t_sel[pe_h] if pe_h is not None else t_sel[vs_h]) * n_pe
    att_s = per_pair["vs"] * nnz_vs + per_pair.get("pe", per_pair["vs"]) * nnz_pe
    total_s = sel_s + att_s
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    sample = (f"oracle selection of head {vs_h} (VS) and head {pe_h} (PE) in full "
              f"({t_sel[vs_h]:.2f} s, {t_sel.get(pe_h, 0):.2f} s); " + "; ".join(desc) +
              f"; extrapolated per block pair to {n_vs} VS + {n_pe} PE heads with "
              f"{nnz_vs} VS and {nnz_pe} PE block pairs")
    return {"value": total_s * 1e3, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": sample, "extrapolated": True,
            "measured_s": sum(t_sel.values()) + t_att_total}


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
        nnz = {}
        for kind, h, mult in (("vs", vs_h, w.hq - n_pe), ("pe", pe_h, n_pe)):
            q = O.bf16_bits_to_f64(g["q"][h])
            k = O.bf16_bits_to_f64(g["k"][h // w.group])
            r = O.crisp_select_head(q, k, **params)
            nnz[kind] = int(np.tril(r["mask"]).sum()) * mult
        stats = {"n_vs": w.hq - n_pe, "n_pe": n_pe, "nnz": nnz["vs"] + nnz["pe"],
                 "nnz_vs": nnz["vs"], "nnz_pe": nnz["pe"]}
        cb = cpu_oracle_sample(w, g, stats, budget_s=args.ref_budget)
        if step >= args.warmup:
            vals.append(cb["value"])
    value = statistics.mean(vals)
    cb["value"] = value
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": value, "higher_is_better": False, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (planted, seeded)",
            "config": dict(workload_config(w), vs_variant=args.vs_variant), "cpu_baseline": cb,
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


def route_pair_counts(ctx, dims, nb):
    """Selected block pairs of the context's selection on VS-routed and PE-routed heads."""
    sel = ctx.selection_get(dims, with_csr=False)
    rp = sel["row_ptr"]
    per_head = rp[nb::nb] - rp[:-1:nb]
    vs = sel["route_vs"].astype(bool)
    return int(per_head[vs].sum()), int(per_head[~vs].sum())


def timed_steps(ctx, dims, q, k, v, o, cfg, steps, stream):
    """`steps` back-to-back crisp_select + crisp_attend on `stream` (CUDA events):
    (total ms, mean select ms, mean attend ms)."""
    import torch
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(steps):
        ev[i][0].record(stream)
        ctx.select(dims, q, k, cfg)
        ev[i][1].record(stream)
        ctx.attend(dims, q, k, v, o)
        ev[i][2].record(stream)
    t1.record(stream)
    torch.cuda.synchronize()
    return (t0.elapsed_time(t1), statistics.mean(e[0].elapsed_time(e[1]) for e in ev),
            statistics.mean(e[1].elapsed_time(e[2]) for e in ev))


def timed_dense(ctx, dims, q, k, v, o, steps, stream):
    import torch
    ctx.dense(dims, q, k, v, o)
    torch.cuda.synchronize()
    de = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    de[0].record(stream)
    for _ in range(steps):
        ctx.dense(dims, q, k, v, o)
    de[1].record(stream)
    torch.cuda.synchronize()
    if ctx.sync_status() != 0:
        raise RuntimeError("device error in dense attention")
    return de[0].elapsed_time(de[1]) / steps


def e2e_host(ctx, dims, cfg, g, q, k, v, o, calls, stream):
    """The same layer through crisp_prefill_host from pinned host buffers (uploads of Q, K,
    V and the download of O inside the timed region, overlapped chunk by chunk), `calls`
    calls after one untimed call; plus the copies alone (one H2D of Q, K, V and one D2H of
    O, back to back on the stream) for the achieved copy bandwidth."""
    import torch
    qh = torch.from_numpy(g["q"].view(np.int16)).view(torch.bfloat16).pin_memory()
    kh = torch.from_numpy(g["k"].view(np.int16)).view(torch.bfloat16).pin_memory()
    vh = torch.from_numpy(g["v"].view(np.int16)).view(torch.bfloat16).pin_memory()
    oh = torch.empty(o.shape, dtype=torch.bfloat16).pin_memory()
    h2d = int(qh.numel() + kh.numel() + vh.numel()) * 2
    d2h = int(oh.numel()) * 2
    ctx.prefill_host(dims, qh, kh, vh, cfg, oh, q, k, v, o)
    torch.cuda.synchronize()
    per_call = []
    for _ in range(calls):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        ctx.prefill_host(dims, qh, kh, vh, cfg, oh, q, k, v, o)
        e1.record(stream)
        torch.cuda.synchronize()
        per_call.append(e0.elapsed_time(e1))
    if ctx.sync_status() != 0:
        raise RuntimeError("device error in the end-to-end run")
    c = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    c[0].record(stream)
    q.copy_(qh, non_blocking=True)
    k.copy_(kh, non_blocking=True)
    v.copy_(vh, non_blocking=True)
    c[1].record(stream)
    oh.copy_(o, non_blocking=True)
    c[2].record(stream)
    torch.cuda.synchronize()
    h2d_ms, d2h_ms = c[0].elapsed_time(c[1]), c[1].elapsed_time(c[2])
    del qh, kh, vh, oh
    return {"per_call_ms": per_call, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "h2d_gbs": h2d / (h2d_ms * 1e-3) / 1e9, "d2h_gbs": d2h / (d2h_ms * 1e-3) / 1e9,
            "copies_alone_ms": h2d_ms + d2h_ms}


def point_128k(dsp, w, g, steps, warmup, dense_steps, dev, stream):
    """select, attend and layer ms, effective TFLOP/s and the dense speedup of one 128k
    workload (device-resident inputs, same timing as the headline)."""
    import torch

    def dev_tensor(u16):
        return torch.from_numpy(u16.view(np.int16)).view(torch.bfloat16).to(dev)

    q, k, v = dev_tensor(g["q"]), dev_tensor(g["k"]), dev_tensor(g["v"])
    o = torch.empty_like(q)
    dims = dsp.make_dims(1, w.n, w.hq, w.hkv)
    ctx = dsp.Context(dims)
    cfg = dsp.default_cfg(alpha=w.alpha, gamma=w.gamma, tau_proxy=w.tau_proxy,
                          k_min_tokens=w.k_min_tokens)
    for _ in range(warmup):
        ctx.prefill(dims, q, k, v, cfg, o)
    if ctx.sync_status() != 0:
        raise RuntimeError(f"device error during warm-up of {w.name}")
    st = ctx.stats(dims)
    total, sel_ms, att_ms = timed_steps(ctx, dims, q, k, v, o, cfg, steps, stream)
    if ctx.sync_status() != 0:
        raise RuntimeError(f"device error in {w.name}")
    dense_ms = timed_dense(ctx, dims, q, k, v, o, dense_steps, stream)
    ctx.close()
    nbk = w.n // B
    flops = algorithmic_flops(st["nnz"], st["rows"])
    ms = total / steps
    return {"n": w.n, "hq": w.hq, "hkv": w.hkv, "alpha": w.alpha, "ms_per_layer": ms,
            "select_ms": sel_ms, "attend_ms": att_ms,
            "tflops_effective": flops / (ms * 1e-3) / 1e12,
            "attend_tflops": flops / (att_ms * 1e-3) / 1e12, "dense_ms": dense_ms,
            "dense_tflops": algorithmic_flops(w.hq * nbk * (nbk + 1) // 2, w.hq * nbk)
            / (dense_ms * 1e-3) / 1e12,
            "speedup_vs_dense": dense_ms / ms,
            "density": st["nnz"] / (w.hq * nbk * (nbk + 1) / 2),
            "n_vs": st["n_vs"], "n_pe": st["n_pe"], "steps": steps, "warmup": warmup}


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
    stats["nnz_vs"], stats["nnz_pe"] = route_pair_counts(ctx, dims, w.n // B)

    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(dev.index) as clk:
        total_ms, sel_ms, att_ms = timed_steps(ctx, dims, q, k, v, o, cfg, args.steps, stream)
    if world > 1:
        dist.barrier()
    if ctx.sync_status() != 0:
        raise RuntimeError("device error during the timed region")
    total_ms = max_over_ranks(total_ms)
    ms_per_step = total_ms / args.steps
    value = replica_value(ms_per_step, world)

    # end to end through the public API with host buffers (pinned), copies included
    e2e = e2e_host(ctx, dims, cfg, g, q, k, v, o, max(5, min(args.steps, 8)), stream)
    e2e_ms = statistics.mean(e2e["per_call_ms"])

    # dense causal attention on the same inputs (the speedup denominator)
    dense_ms = None if args.no_dense else timed_dense(ctx, dims, q, k, v, o, args.dense_steps,
                                                      stream)
    ctx.close()
    del q, k, v, o

    # the metric's 128k point: the Llama-3-8B layer at alpha = 1.0 and 1.25, and the
    # Qwen2-7B layer, each after the headline's timed region
    at_128k = None
    if not args.no_128k:
        from workloads import get
        at_128k = {}
        g128 = None
        for name in ("llama8b_n128k_a1", "llama8b_n128k_a125", "qwen7b_n128k"):
            w1 = get(name)
            if g128 is None or g128[0] != (w1.seed, w1.hq, w1.hkv, w1.n):
                g128 = ((w1.seed, w1.hq, w1.hkv, w1.n), make_inputs(w1))
            at_128k[name] = point_128k(dsp, w1, g128[1], args.steps_128k, 2,
                                       args.dense_steps, dev, stream)
        del g128
        torch.cuda.empty_cache()

    if rank != 0:
        return
    peaks, peak_kind = load_peaks()
    flops = algorithmic_flops(stats["nnz"], stats["rows"])
    att_tflops = flops / (att_ms * 1e-3) / 1e12
    peak = float(peaks.get("bf16_tflops_sustained", peaks.get("bf16_tflops")))
    clocks = clk.summary()
    peak_mhz = (peaks.get("clocks_under_load") or {}).get("sm_mhz_median")
    run_mhz = clocks.get("sm_mhz")
    nbk = w.n // B
    dense_flops = algorithmic_flops(w.hq * nbk * (nbk + 1) // 2, w.hq * nbk)
    roofline = {
        "kernel": "attention_kernel", "bound": "tensor", "achieved": att_tflops,
        "peak": peak, "unit": "TFLOP/s", "frac": att_tflops / peak,
        "peak_kind": f"bf16 sustained (cuBLAS, seconds-long loop), {peak_kind}",
        "unit_of_work": "one crisp_attend call (all launches of the attention kernels for "
                        "the layer)",
        "algorithmic_flops_per_attend": flops,
        "traffic": None,
        "traffic_note": "null: this run counts no DRAM bytes, and counter captures at this "
                        "size are limited to durations. Small-case captures do not scale: one "
                        "32k launch reads 1.33x its algorithmic bytes, one 512k launch "
                        "(a KV head, reduced-head workload) about 7x, from L2 misses as "
                        "its CTAs spread over the KV head's K/V",
    }
    if peak_mhz and run_mhz:
        # the measured peak was taken at its own median SM clock; scaled to this run's
        roofline["peak_sm_mhz"] = peak_mhz
        roofline["run_sm_mhz"] = run_mhz
        roofline["peak_at_run_clock"] = peak * run_mhz / peak_mhz
        roofline["frac_at_run_clock"] = att_tflops / roofline["peak_at_run_clock"]
        roofline["frac_basis"] = ("frac: against the measured sustained peak as recorded; "
                                  "frac_at_run_clock: that peak scaled by this run's median "
                                  "SM clock over the peak's")
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
                      "nnz_vs": stats["nnz_vs"], "nnz_pe": stats["nnz_pe"],
                      "pe_rescued_rows": stats["pe_rescued"], "max_row": stats["max_row"]},
        "roofline": roofline,
        "gpu_launches": launches_per_prefill(w, torch.cuda.get_device_properties(0).multi_processor_count) * args.steps,
        "e2e": {"value": e2e_ms / world, "unit": UNIT,
                "h2d_bytes_per_step": e2e["h2d_bytes_per_step"],
                "d2h_bytes_per_step": e2e["d2h_bytes_per_step"],
                "calls": len(e2e["per_call_ms"]),
                "per_call_ms": [round(x, 2) for x in e2e["per_call_ms"]],
                "h2d_gbs": e2e["h2d_gbs"], "d2h_gbs": e2e["d2h_gbs"],
                "copies_alone_ms": e2e["copies_alone_ms"],
                "exposed_over_device_ms": e2e_ms - ms_per_step},
        "clocks": clocks,
        "at_128k": at_128k,
        "pages_context": {"crisp_speedup_vs_flashattention_512k_h100": 5.30},
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_oracle_sample(w, g, stats, budget_s=args.ref_budget)
    print(json.dumps(line), flush=True)


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
    ap.add_argument("--no-128k", action="store_true",
                    help="skip the 128k points (Llama alpha 1.0 / 1.25, Qwen) after the headline")
    ap.add_argument("--steps-128k", type=int, default=5)
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
