"""Benchmark of the paged fused-MoE layer forward on GB300.

One step = one forward of the Mixtral-8x7B-shaped layer (d=4096, f=14336, 8 experts top-2; 6
experts in random pool pages, 2 in a load buffer; logits with +1.0 on two hot experts) over a
batch of T=8192 synthetic tokens, the largest workload of the set, with weights, tables and
activations resident in HBM.  The JSON line reports TFLOP/s (algorithmic: 6*T*d*(k*f + S*f)),
the same through host buffers (e2e), the dominant kernel against its roofline (the burst bf16
peak unless the timed region lasts 2 s or more), the paged-vs-contiguous overhead, token-count
sweeps, the CPU oracle's throughput on a bounded sample of the same workload, and the
Qwen1.5-MoE- and Qwen3-Next-shaped layers at 4096 tokens with their sweeps as extra keys.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--config mixtral] [--tokens 8192] [--no-sweep] [--no-cpu] [--no-extra]

Under torchrun every rank runs its own replica (the path has no collective); rank 0 prints.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from paged_moe_expert_gb300 import synthetic as syn  # noqa: E402

METRIC = "paged fused-MoE TFLOP/s & weight GB/s vs roofline; overhead vs contiguous"
PATH_NAMES = {0: "auto", 1: "stream", 2: "tc", 3: "tc_decode", 4: "tc2", 5: "fused", 6: "slice"}
L2_BYTES = 129 * 2 ** 20


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                "sm_max_mhz": d.get("sm_max_mhz", 2070.0), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "sm_max_mhz": 2070.0, "source": "fallback"}


# ---------------------------------------------------------------------------------------------
# algorithmic work
# ---------------------------------------------------------------------------------------------

def work(cfg, T, e_act):
    """Algorithmic FLOPs and bytes of one forward, and of its two GEMM kernels."""
    d, f, k, S, E = cfg.d, cfg.f, cfg.k, cfg.S, cfg.E
    pairs = T * (k + S)
    flops = 6.0 * T * d * (k * f + S * f)
    wbytes = 6.0 * d * f * (e_act + S)
    total_bytes = wbytes + 4.0 * T * d + 4.0 * T * E
    g1 = {"flops": 4.0 * pairs * d * f, "bytes": 4.0 * d * f * (e_act + S) + 2.0 * pairs * (d + f)}
    g2 = {"flops": 2.0 * pairs * d * f,
          "bytes": 2.0 * d * f * (e_act + S) + 2.0 * pairs * f + 2.0 * pairs * d}   # bf16 h in, y out
    return {"flops": flops, "weight_bytes": wbytes, "bytes": total_bytes, "gemm1": g1, "gemm2": g2}


# the committed ncu summary and the source file of each profiled kernel, by (path, kernel)
PROFILED = {("tc", "gemm1"): ("tc_gemm", "tc_gemm.cu"), ("tc", "gemm2"): ("tc_gemm", "tc_gemm.cu"),
            ("tc2", "gemm1"): ("tc_gemm2sm", "tc_gemm2sm.cu"),
            ("tc2", "gemm2"): ("tc_gemm2sm", "tc_gemm2sm.cu"),
            ("fused", "fused"): ("fused_decode", "tc_fused.cu")}


def measured_traffic(cfg_key, T, path_name, kernel):
    """DRAM traffic per launch (read + write bytes) of `kernel` from the committed ncu summary of
    this workload, or None when there is none or the kernel source changed since it was taken."""
    import hashlib
    if (path_name, kernel) not in PROFILED:
        return None
    prefix, srcname = PROFILED[(path_name, kernel)]
    path = os.path.join(ROOT, "profiles", "%s_%s_T%d.md" % (prefix, cfg_key, T))
    if not os.path.exists(path):
        return None
    fields = {}
    for line in open(path):
        if ":" in line and line.startswith("traffic_"):
            k, v = line.split(":", 1)
            fields[k.strip()] = v.strip()
    src = os.path.join(ROOT, "paged_moe_expert_gb300", "csrc", srcname)
    sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    if fields.get("traffic_source_sha256_prefix", sha) != sha:
        return None
    v = fields.get("traffic_%s_bytes_per_launch" % kernel)
    return int(v) if v else None


def binding_fraction(flops, nbytes, seconds, peaks, sustained=True):
    tc = peaks["bf16_tflops_sustained" if sustained else "bf16_tflops"] * 1e12
    bw = peaks["hbm_gbs"] * 1e9
    t_roof = max(flops / tc, nbytes / bw)
    return t_roof / seconds, ("tensor" if flops / tc > nbytes / bw else "hbm")


# ---------------------------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------------------------

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,utilization.gpu,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.dev = device_index
        self.p = None
        self.path = os.path.join("/tmp", "pmoe_clocks_%d_%d.csv" % (os.getpid(), device_index))

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(self.dev), "--query-gpu=" + self.QUERY,
                                       "--format=csv,noheader,nounits", "-lms", "200"],
                                      stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.p = None

    def stop(self):
        if self.p is None:
            return None
        self.p.terminate()
        try:
            self.p.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.p.kill()
        self.f.close()
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                rows.append({"sm": float(parts[1]), "max": float(parts[2]), "util": float(parts[4]),
                             "hw_slowdown": parts[6], "hw_thermal": parts[7], "sw_thermal": parts[8],
                             "sw_power_cap": parts[9]})
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return None
        loaded = [r for r in rows if r["util"] >= 50] or rows
        reasons = set()
        for r in loaded:
            for key in ("hw_slowdown", "hw_thermal", "sw_thermal", "sw_power_cap"):
                if r[key].lower() == "active":
                    reasons.add({"hw_thermal": "hw_thermal_slowdown", "sw_thermal": "sw_thermal_slowdown"}.get(key, key))
        return {"sm_mhz": statistics.median(r["sm"] for r in loaded),
                "sm_max_mhz": max(r["max"] for r in loaded), "reasons": sorted(reasons),
                "samples": len(loaded)}


# ---------------------------------------------------------------------------------------------
# the CPU oracle (baseline / reference arm)
# ---------------------------------------------------------------------------------------------

def oracle_throughput(cfg, w, hidden, logits, budget_s, max_tokens):
    """Time the oracle, as it stands, on the first n tokens of the batch; n is sized from a
    short calibration run so the timed run takes about budget_s seconds."""
    import oracle
    L = oracle.Layer(w.W1, w.W3, w.W2, cfg.k, cfg.renormalize, W1s=w.W1s, W3s=w.W3s, W2s=w.W2s, S=cfg.S)
    cores = os.cpu_count() or 1
    n0 = min(max_tokens, cores)
    t0 = time.perf_counter()
    L.forward(hidden[:n0], logits[:n0], nthreads=cores)
    dt = time.perf_counter() - t0
    n = int(min(max_tokens, max(n0, n0 * budget_s / max(dt, 1e-6))))
    n = max(cores, n // cores * cores) if n >= cores else n
    t0 = time.perf_counter()
    L.forward(hidden[:n], logits[:n], nthreads=cores)
    dt = time.perf_counter() - t0
    flops = 6.0 * n * cfg.d * (cfg.k * cfg.f + cfg.S * cfg.f)
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": "first %d of %d tokens of the same batch, all experts, fp64 C oracle, %.2f s"
                      % (n, hidden.shape[0], dt), "tokens": n, "seconds": dt}


def run_reference(args, rank):
    if rank != 0:
        return
    cfg = syn.CONFIGS[args.config]
    T = args.tokens or cfg.tokens[-1]
    w = syn.make_weights(cfg)
    hidden, logits = syn.make_tokens(cfg, T)
    import oracle
    L = oracle.Layer(w.W1, w.W3, w.W2, cfg.k, cfg.renormalize, W1s=w.W1s, W3s=w.W3s, W2s=w.W2s, S=cfg.S)
    cores = os.cpu_count() or 1
    # size one step to about 4 s of CPU work so warmup + steps end within a few minutes
    cal = oracle_throughput(cfg, w, hidden, logits, 2.0, T)
    per_tok = cal["seconds"] / cal["tokens"]
    n = int(max(1, min(T, 4.0 / per_tok)))
    for _ in range(args.warmup):
        L.forward(hidden[:n], logits[:n], nthreads=cores)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        L.forward(hidden[:n], logits[:n], nthreads=cores)
    dt = (time.perf_counter() - t0) / args.steps
    flops = 6.0 * n * cfg.d * (cfg.k * cfg.f + cfg.S * cfg.f)
    v = flops / dt / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": "%s layer forward, T=%d tokens (each step a %d-token sample)"
                       % (cfg.name, T, n), "tokens": T, "sample_tokens": n},
            "cpu_baseline": {"value": v, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                             "sample": "first %d of %d tokens per step" % (n, T)},
            "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------------------------

class Layer:
    def __init__(self, cfg, device, contiguous=True):
        import paged_moe_expert_gb300 as pm
        from paged_moe_expert_gb300 import pool as pl
        self.pm, self.cfg, self.device = pm, cfg, device
        self.w = syn.make_weights(cfg)
        self.placement = syn.make_placement(cfg)
        self.pool = pl.new_pool(cfg.num_pages, cfg.f, cfg.d, device)
        self.bufs = pl.new_load_buffers(cfg.slots_per_buffer, cfg.f, cfg.d, device)
        pt, bs = pl.place(cfg, self.w, self.placement, self.pool, self.bufs, 0)
        self.page_table, self.buf_slot = pt.to(device), bs.to(device)
        self.desc = pm.make_desc(cfg.d, cfg.f, cfg.E, cfg.k, cfg.renormalize, cfg.S,
                                 cfg.slots_per_buffer)
        self.plan = pm.Plan(self.desc, self.pool, cfg.num_pages, self.bufs)
        self.cplan = None
        if contiguous:
            self.cweights = pl.contiguous_weights(cfg, self.w, device)
            self.cplan = pm.Plan(self.desc, self.cweights, 3 * (cfg.E + cfg.S))

    def tokens(self, T):
        from paged_moe_expert_gb300 import pool as pl
        h, lg = syn.make_tokens(self.cfg, T)
        return h, lg, pl._bf16(h).to(self.device), torch.from_numpy(lg).to(self.device)

    def e_act(self, logits_dev):
        ids, _ = self.pm.route(logits_dev, self.cfg.k, self.cfg.renormalize)
        return int(torch.unique(ids).numel())


def tc_family_path(path):
    return path in (2, 3, 4, 5, 6)


def max_over_ranks(seconds: float, dist, device) -> float:
    """The slowest rank's time: every rank's replica must finish before the step is done."""
    if dist is None:
        return seconds
    t = torch.tensor([seconds], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: float, world: int, seconds: float) -> float:
    """Whole-job throughput: the units all ranks processed over the slowest rank's time."""
    return units_per_rank * world / seconds


def capture(fn):
    """fn's launches captured once into a CUDA graph (replayed by the sweep)."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


def time_iters(fn_list, iters, flush):
    """Median device time (s) of each fn, interleaved, L2 flushed before every timed call."""
    times = [[] for _ in fn_list]
    s = torch.cuda.current_stream()
    for _ in range(iters):
        for i, fn in enumerate(fn_list):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(s)
            fn()
            b.record(s)
            b.synchronize()
            times[i].append(a.elapsed_time(b) * 1e-3)
    return [statistics.median(t) for t in times]


def decode_sweep(args):
    """24 consecutive Qwen1.5-MoE-shaped layers per step, batch 1..256 tokens, resident fraction
    100% -> 50%: offloaded experts stream from pinned host memory into the two alternating load
    buffers one layer ahead of compute; the pool layout cycles over 4 pre-placed layouts per step.
    With --predicted the prefetch follows a prediction (each layer's routing in the previous step)
    instead of the actual routing, and each layer first copies in the routed experts the
    prediction missed (pmoe_copy_in_missing), timed as its stall.  One JSON line per (resident
    fraction, tokens)."""
    from paged_moe_expert_gb300 import pipeline
    import paged_moe_expert_gb300 as pm
    torch.cuda.set_device(0)
    cfg = syn.CONFIGS["qwen15"]
    w = syn.make_weights(cfg)
    L = args.layers
    tokens_list = [int(x) for x in args.tokens_list.split(",")]
    fractions = [float(x) for x in args.fractions.split(",")]
    # host -> device copy bandwidth (pinned), for the copy-time estimate
    hbuf = torch.empty(1 << 30, dtype=torch.uint8).pin_memory()
    dbuf = torch.empty(1 << 30, dtype=torch.uint8, device="cuda")
    dbuf.copy_(hbuf, non_blocking=True)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(3):
        dbuf.copy_(hbuf, non_blocking=True)
    b.record()
    torch.cuda.synchronize()
    h2d_gbs = 3 * (1 << 30) / (a.elapsed_time(b) * 1e-3) / 1e9
    del hbuf, dbuf
    if args.predicted and args.backend != "host":
        raise SystemExit("--predicted copies missed experts from pinned host memory: use --backend host")
    resident_ms = {}
    for frac in fractions:
        n_off = int(round((1.0 - frac) * cfg.E))
        stack = pipeline.DecodeStack(cfg, w, L, n_off, layouts=4, seed=11, backend=args.backend)
        for T in tokens_list:
            rng = np.random.default_rng(1000 + T)
            steps = args.warmup + args.steps
            logits = [[syn.bf16_bits_to_f32(syn.to_bf16_bits(
                rng.standard_normal((T, cfg.E)).astype(np.float32))) for _ in range(L)]
                for _ in range(steps)]
            n_missed = 0
            if args.predicted:
                # prediction for step s = each layer's routing in step s - 1 (a step before the first)
                before = [syn.bf16_bits_to_f32(syn.to_bf16_bits(
                    rng.standard_normal((T, cfg.E)).astype(np.float32))) for _ in range(L)]
                preds = [[pipeline.routed_experts((logits[s_ - 1] if s_ else before)[l], cfg.k)
                          for l in range(L)] for s_ in range(steps)]
                scheds = [stack.schedule_predicted(p_) for p_ in preds]
                n_missed = sum(len(np.setdiff1d(np.intersect1d(pipeline.routed_experts(logits[s_][l], cfg.k),
                                                               stack.offloaded[l]), preds[s_][l]))
                               for s_ in range(args.warmup, steps) for l in range(L))
            else:
                scheds = [stack.schedule(lg) for lg in logits]
            lg_dev = [[torch.from_numpy(x).cuda() for x in lg] for lg in logits]
            stall = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                      for _ in range(L)] for _ in range(args.steps)] if args.predicted else None
            hidden = torch.from_numpy(syn.to_bf16_bits(rng.standard_normal((T, cfg.d)).astype(
                np.float32)).view(np.int16)).view(torch.bfloat16).cuda()
            ws = pm.alloc_workspace(stack.desc, T)
            acts = [torch.empty_like(hidden) for _ in range(2)]
            n_pref = sum(len(sc[0]) for sched in scheds[args.warmup:] for sc in sched)
            copied = (n_pref + n_missed) * 6 * cfg.d * cfg.f
            for s_ in range(args.warmup):
                stack.step(hidden, lg_dev[s_], scheds[s_], s_, acts, ws, copy_in=args.predicted)
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for s_ in range(args.warmup, steps):
                stack.step(hidden, lg_dev[s_], scheds[s_], s_, acts, ws, copy_in=args.predicted,
                           stall_events=stall[s_ - args.warmup] if stall else None)
            e1.record()
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1) / args.steps
            for row in stack.plans:
                for p_ in row:
                    if p_.device_error() != 0:
                        raise RuntimeError("device error word set in the decode sweep")
            stall_ms = (sum(a_.elapsed_time(b_) for st in stall for a_, b_ in st) / args.steps
                        if stall else None)
            if n_off == 0:
                resident_ms[T] = ms
            copy_ms = copied / args.steps / (h2d_gbs * 1e9) * 1e3 if args.backend == "host" else 0.0
            line = {"metric": "decode sweep: 24-layer step time with double-buffered expert prefetch",
                    "config": {"workload": "%d Qwen1.5-MoE-shaped layers, %d tokens/step" % (L, T),
                               "resident_fraction": frac, "offloaded_experts_per_layer": n_off,
                               "pool_layouts_cycled": 4,
                               "offload_backend": ("pinned host memory" if args.backend == "host" else
                                                   "exponent-Huffman blobs in device memory")},
                    "tokens": T, "ms_per_step": ms, "tokens_per_s": T / (ms * 1e-3),
                    "copied_mb_per_step": copied / args.steps / 1e6,
                    "h2d_gbs": h2d_gbs, "copy_ms_per_step_est": copy_ms,
                    "all_resident_ms": resident_ms.get(T),
                    "prefetch": ("previous step's routing (copy-in of misses)" if args.predicted
                                 else "actual routing"),
                    "experts_prefetched_per_step": n_pref / args.steps,
                    "experts_copied_in_per_step": n_missed / args.steps,
                    "copy_in_ms_per_step": stall_ms,
                    "exposed_copy_frac": (None if T not in resident_ms or copy_ms == 0 else
                                          max(0.0, (ms - resident_ms[T])) / copy_ms)}
            print(json.dumps(line), flush=True)
            del ws, acts
        del stack
        torch.cuda.empty_cache()


def vmm_overhead(args):
    """The page lookup against the rival remapped view (FluxMoE's PagedTensor: physical blocks
    mapped under stable virtual addresses with the CUDA driver's VMM calls, the contiguous kernel
    unchanged) and against an ordinary contiguous allocation, on the layer shapes whose expert
    page is a whole number of VMM blocks.  All experts resident, the page table a random
    permutation of the blocks; CUDA-graph replay, L2 flushed before every timed call.  One JSON
    line per (layer, tokens)."""
    import paged_moe_expert_gb300 as pm
    from paged_moe_expert_gb300 import pool as pl
    from paged_moe_expert_gb300 import vmm as vm
    torch.cuda.set_device(0)
    device = torch.device("cuda", 0)
    g = vm.granularity(0)
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=device)
    for cname in ("qwen3next", "mixtral", "qwen15"):
        cfg = syn.CONFIGS[cname]
        E, S, f, d = cfg.E, cfg.S, cfg.f, cfg.d
        page = f * d * 2
        if page % g:
            print(json.dumps({"metric": "remapped view vs page lookup", "config": {"workload": cfg.name},
                              "skipped": "expert page of %d bytes is not a multiple of the %d-byte VMM "
                                         "granularity" % (page, g)}), flush=True)
            continue
        w = syn.make_weights(cfg)
        n = 3 * (E + S)
        v = vm.VmmView(page, n, n)
        pt = np.random.default_rng(5).permutation(n).astype(np.int32).reshape(E + S, 3)
        desc = pm.make_desc(d, f, E, cfg.k, cfg.renormalize, S, 1)
        plan_b = pm.Plan(desc, v.blocks, n)
        host = [torch.from_numpy(pl.pack_expert(w, e, E, f).view(np.int16)).pin_memory()
                for e in range(E + S)]
        cs = torch.cuda.Stream()
        pm.fill_pages_async(plan_b, host, pt.tolist(), cs)
        cs.synchronize()
        del host
        vm.map_experts(v, pt)
        assert (v.lookup() >= 0).all()
        plan_v = pm.Plan(desc, v.view, n)
        cw = pl.contiguous_weights(cfg, w, device)
        plan_c = pm.Plan(desc, cw, n)
        ptd = torch.from_numpy(pt).to(device)
        bs = torch.full((E,), -1, dtype=torch.int32, device=device)
        for T in cfg.tokens:
            h, lg = syn.make_tokens(cfg, T)
            hd, ld = pl._bf16(h).to(device), torch.from_numpy(lg).to(device)
            ws = pm.alloc_workspace(desc, T, device)
            o = torch.empty_like(hd)
            fp = lambda: plan_b.forward(hd, ld, ptd, bs, out=o, workspace=ws)  # noqa: E731
            fv = lambda: plan_v.contig_forward(hd, ld, out=o, workspace=ws)  # noqa: E731
            fc = lambda: plan_c.contig_forward(hd, ld, out=o, workspace=ws)  # noqa: E731
            for _ in range(3):
                fp(); fv(); fc()
            path = plan_b.last_run()[0]
            gp, gv, gc = capture(fp), capture(fv), capture(fc)
            tp, tv, tc = time_iters([gp.replay, gv.replay, gc.replay], args.sweep_iters, flush)
            assert plan_b.device_error() == 0
            print(json.dumps({
                "metric": "remapped view vs page lookup",
                "config": {"workload": "%s layer forward, T=%d tokens, all experts resident, "
                           "pages scattered over %d blocks of %d bytes" % (cfg.name, T, n, page)},
                "path": PATH_NAMES[path], "paged_ms": tp * 1e3, "remapped_view_ms": tv * 1e3,
                "contiguous_alloc_ms": tc * 1e3, "paged_vs_view": tp / tv - 1.0,
                "paged_vs_alloc": tp / tc - 1.0, "view_vs_alloc": tv / tc - 1.0}), flush=True)
            del ws, o
        del plan_v, plan_b, plan_c, cw
        v.close()
        torch.cuda.empty_cache()


def codec_bench(args):
    """Exponent-only Huffman pages (FluxMoE's compressed GPU backend): the buffered experts of the
    Qwen1.5-MoE-shaped layer (15 experts, 45 pages) encoded on the host, decoded on the GPU into a
    load buffer in one launch; against copying the same pages uncompressed from pinned host
    memory.  One JSON line."""
    import paged_moe_expert_gb300 as pm
    from paged_moe_expert_gb300 import expcodec as nc
    from paged_moe_expert_gb300 import pool as pl
    torch.cuda.set_device(0)
    cfg = syn.CONFIGS["qwen15"]
    w = syn.make_weights(cfg)
    E, f, d = cfg.E, cfg.f, cfg.d
    page = f * d
    n_exp = cfg.n_buffered
    mats = [m for e in range(n_exp) for m in pl.expert_matrices(w, e, E, f)]
    t0 = time.time()
    blobs_h = [nc.encode(m) for m in mats]
    enc_s = time.time() - t0
    comp = sum(b.size for b in blobs_h)
    blobs = [torch.from_numpy(b).cuda() for b in blobs_h]
    buf = torch.empty(len(mats) * page, dtype=torch.bfloat16, device="cuda")
    dsts = [buf[i * page:(i + 1) * page] for i in range(len(mats))]
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _ in range(3):
        nc.decode_async(blobs, page, dsts, device_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ok = all(np.array_equal(dsts[i].cpu().view(torch.int16).numpy().view(np.uint16), mats[i].reshape(-1))
             for i in (0, len(mats) - 1))
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device="cuda")
    times = []
    for _ in range(args.sweep_iters):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        nc.decode_async(blobs, page, dsts)
        b.record()
        b.synchronize()
        times.append(a.elapsed_time(b) * 1e-3)
    dec = statistics.median(times)
    host = torch.from_numpy(np.concatenate([m.reshape(-1) for m in mats]).view(np.int16)).pin_memory()
    raw = len(mats) * page * 2
    h2d = []
    for _ in range(5):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        buf.view(torch.int16).copy_(host, non_blocking=True)
        b.record()
        b.synchronize()
        h2d.append(a.elapsed_time(b) * 1e-3)
    h2d_s = statistics.median(h2d)
    print(json.dumps({
        "metric": "exponent-only Huffman decode of bf16 expert pages",
        "config": {"workload": "%d Qwen1.5-MoE-shaped expert pages (%d experts x W1, W3, W2), "
                   "%d bf16 values each, one launch, L2 flushed" % (len(mats), n_exp, page)},
        "compressed_ratio": comp / raw, "encode_host_s": enc_s,
        "decode_ms": dec * 1e3, "decoded_gbs": raw / dec / 1e9,
        "decode_hbm_traffic_gbs": (raw + comp) / dec / 1e9,
        "h2d_uncompressed_ms": h2d_s * 1e3, "h2d_gbs": raw / h2d_s / 1e9, "bit_exact": ok}), flush=True)


def elastic_requests(args):
    """The elastic stack with KV cache pages in the same pool: requests arrive and leave (a
    seeded trace whose arrival rate rises and falls), each holding KV pages of 1/8 expert page
    carved from expert pages the adjuster lends; requests that do not fit wait for a later round.
    24 Qwen1.5-MoE-shaped layers, 16 tokens per step.  One JSON line per phase."""
    from paged_moe_expert_gb300 import pipeline
    import paged_moe_expert_gb300 as pm
    torch.cuda.set_device(0)
    cfg = syn.CONFIGS["qwen15"]
    w = syn.make_weights(cfg)
    L, T, E = args.layers, args.elastic_tokens, cfg.E
    rng = np.random.default_rng(29)
    bias = rng.standard_normal((L, E)).astype(np.float32)

    def draw(n):
        return [syn.bf16_bits_to_f32(syn.to_bf16_bits(
            rng.standard_normal((n, E)).astype(np.float32) + bias[l])) for l in range(L)]

    sample = draw(4096)
    probs = np.stack([np.bincount(np.argsort(-lg, axis=1, kind="stable")[:, :cfg.k].ravel(),
                                  minlength=E) / (4096.0 * cfg.k) for lg in sample]).astype(np.float32)
    expert_pages = 3 * E * L + 3 * 4
    stack = pipeline.ElasticDecodeStack(cfg, w, L, probs, [E] * L, args.offload_limit, expert_pages,
                                        backend=args.backend)
    page_bytes = cfg.f * cfg.d * 2
    kv = pipeline.KVPages(stack.adj, expert_pages, page_bytes, page_bytes // 8)
    hidden = torch.from_numpy(syn.to_bf16_bits(rng.standard_normal((T, cfg.d)).astype(
        np.float32)).view(np.int16)).view(torch.bfloat16).cuda()
    ws = pm.alloc_workspace(stack.desc, T)
    acts = [torch.empty_like(hidden) for _ in range(2)]
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    phases = [("quiet", 10, 0.5), ("arrivals rise", 25, 6.0), ("busy", 25, 6.0),
              ("arrivals fall", 25, 1.0), ("quiet again", 25, 0.2)]
    live_until, waiting, nxt, rnd = {}, {}, 0, 0
    for name, rounds, rate in phases:
        rec = {"ms": [], "kv_pages": [], "waiting": [], "resident": [], "adds": 0, "evicts": 0}
        for _ in range(rounds):
            departures = [r for r, end in live_until.items() if end <= rnd]
            for r in departures:
                del live_until[r]
            arrivals = dict(waiting)
            for _ in range(int(rng.poisson(rate))):
                arrivals[nxt] = int(rng.integers(8, 65))
                nxt += 1
            f0 = stack.filled_experts
            changes, short, waiting = stack.round_requests(kv, arrivals, departures)
            for r in arrivals:
                if r not in waiting:
                    live_until[r] = rnd + int(rng.integers(3, 16))
            lg = draw(T)
            sched = stack.schedule(lg)
            lg_dev = [torch.from_numpy(x).cuda() for x in lg]
            a.record()
            stack.step(hidden, lg_dev, sched, acts, ws)
            b.record()
            torch.cuda.synchronize()
            rec["ms"].append(a.elapsed_time(b))
            rec["kv_pages"].append(sum(len(v) for v in kv.live().values()))
            rec["waiting"].append(len(waiting))
            rec["resident"].append(int(stack.adj.cached().sum()))
            rec["adds"] += stack.filled_experts - f0
            rec["evicts"] += int((changes[:, 0] == -1).sum()) if len(changes) else 0
            rnd += 1
        print(json.dumps({
            "metric": "elastic decode with KV pages in the expert pool: request-driven rounds",
            "config": {"workload": "%d Qwen1.5-MoE-shaped layers, %d tokens/step, KV page = 1/8 "
                       "expert page, %d expert pages, offload limit %d" % (L, T, expert_pages,
                                                                           args.offload_limit),
                       "phase": name, "rounds": rounds, "arrivals_per_round": rate},
            "ms_per_step_median": float(np.median(rec["ms"])),
            "ms_per_step_max": float(np.max(rec["ms"])),
            "kv_pages_end": rec["kv_pages"][-1], "kv_pages_max": max(rec["kv_pages"]),
            "requests_waiting_max": max(rec["waiting"]),
            "resident_experts": [min(rec["resident"]), max(rec["resident"])],
            "experts_added": rec["adds"], "experts_evicted": rec["evicts"]}), flush=True)


def elastic_sweep(args):
    """24 Qwen1.5-MoE-shaped layers on ONE page pool shared with the KV cache.  A KV demand
    trace (in expert pages) rises and falls over the rounds; each round the KV pages are taken
    first and the adjuster evicts or adds experts by the offline ranking (routing frequencies
    measured on a sample drawn from the same skewed router), added experts are copied into their
    reserved pages, and offloaded experts that the step routes to stream through the two load
    buffers.  Prints one JSON line per phase of the trace."""
    from paged_moe_expert_gb300 import pipeline
    import paged_moe_expert_gb300 as pm
    torch.cuda.set_device(0)
    cfg = syn.CONFIGS["qwen15"]
    w = syn.make_weights(cfg)
    L, T, E = args.layers, args.elastic_tokens, cfg.E
    rng = np.random.default_rng(23)
    bias = rng.standard_normal((L, E)).astype(np.float32)     # per-layer expert popularity

    def draw(n):
        return [syn.bf16_bits_to_f32(syn.to_bf16_bits(
            rng.standard_normal((n, E)).astype(np.float32) + bias[l])) for l in range(L)]

    sample = draw(4096)   # "offline" profiling sample -> routing probability per expert
    probs = np.stack([np.bincount(np.argsort(-lg, axis=1, kind="stable")[:, :cfg.k].ravel(),
                                  minlength=E) / (4096.0 * cfg.k) for lg in sample]).astype(np.float32)
    limit = args.offload_limit
    expert_pages = 3 * E * L + 3 * 4
    stack = pipeline.ElasticDecodeStack(cfg, w, L, probs, [E] * L, limit, expert_pages,
                                        backend=args.backend)
    peak = args.kv_peak
    phases = [("idle, all experts resident", [0] * 5),
              ("KV demand ramps up", [int(peak * (i + 1) / 20) for i in range(20)]),
              ("KV demand held at peak", [peak] * 20),
              ("KV demand ramps down", [int(peak * (19 - i) / 20) for i in range(20)]),
              ("idle again", [0] * 25)]
    hidden = torch.from_numpy(syn.to_bf16_bits(rng.standard_normal((T, cfg.d)).astype(
        np.float32)).view(np.int16)).view(torch.bfloat16).cuda()
    ws = pm.alloc_workspace(stack.desc, T)
    acts = [torch.empty_like(hidden) for _ in range(2)]
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    page_mb = cfg.f * cfg.d * 2 / 1e6
    for name, trace in phases:
        rec = {"ms": [], "resident": [], "kv_pages": [], "short": [], "adds": 0, "evicts": 0,
               "prefetched": 0}
        for need in trace:
            lg = draw(T)
            f0 = stack.filled_experts
            changes, short = stack.round(need)
            sched = stack.schedule(lg)
            lg_dev = [torch.from_numpy(x).cuda() for x in lg]
            a.record()
            stack.step(hidden, lg_dev, sched, acts, ws)
            b.record()
            torch.cuda.synchronize()
            rec["ms"].append(a.elapsed_time(b))
            rec["resident"].append(int(stack.adj.cached().sum()))
            rec["kv_pages"].append(len(stack.kv))
            rec["short"].append(int(short))
            rec["adds"] += stack.filled_experts - f0
            rec["evicts"] += int((changes[:, 0] == -1).sum()) if len(changes) else 0
            rec["prefetched"] += sum(len(sc[0]) for sc in sched)
        n = len(trace)
        line = {"metric": "elastic decode: adjuster-driven 24-layer step on one pool shared with KV",
                "config": {"workload": "%d Qwen1.5-MoE-shaped layers, %d tokens/step, %d expert "
                           "pages (%.2f MB each), offload limit %d" % (L, T, expert_pages, page_mb, limit),
                           "phase": name, "rounds": n, "kv_demand_pages": [trace[0], trace[-1]],
                           "offload_backend": ("pinned host memory" if args.backend == "host" else
                                               "exponent-Huffman blobs in device memory")},
                "ms_per_step_median": float(np.median(rec["ms"])),
                "ms_per_step_max": float(np.max(rec["ms"])),
                "tokens_per_s": T / (float(np.median(rec["ms"])) * 1e-3),
                "resident_experts": [min(rec["resident"]), max(rec["resident"])],
                "kv_pages_held_end": rec["kv_pages"][-1], "short_pages_max": max(rec["short"]),
                "experts_added": rec["adds"], "experts_evicted": rec["evicts"],
                "experts_streamed_per_step": rec["prefetched"] / n,
                "copied_mb_per_step": (rec["adds"] + rec["prefetched"]) * 3 * page_mb / n}
        print(json.dumps(line), flush=True)


PATH_IDS = {"auto": 0, "stream": 1, "tc": 2, "tc_decode": 3, "tc2": 4, "fused": 5, "slice": 6}
# a timed region at least this long runs at the power-capped (sustained) clocks; shorter ones are
# compared with the burst peak
SUSTAINED_REGION_S = 2.0


def kernel_names(nk, path):
    if nk == 6:
        return ["route", "align", "gather", "gemm1", "gemm2", "combine"]
    if nk == 5:
        return (["prep", "gather"] if tc_family_path(path) else ["route", "align"]) + ["gemm1", "gemm2", "combine"]
    if nk == 1:
        return ["fused"]   # routing, both projections and the combine in one kernel
    return ["prep", "gemm1", "gemm2", "combine"]


def dominant_roofline(kwork, ksec, path, peaks, region_s):
    """The dominant kernel against the roof that binds it.  Tensor-bound kernels take the burst
    bf16 peak unless the timed region is long enough to run at sustained (power-capped) clocks."""
    sustained = region_s >= SUSTAINED_REGION_S
    tc_peak = peaks["bf16_tflops_sustained" if sustained else "bf16_tflops"]
    tc_family = tc_family_path(path)
    if tc_family and kwork["flops"] / (tc_peak * 1e12) > kwork["bytes"] / (peaks["hbm_gbs"] * 1e9):
        roof = {"bound": "tensor", "achieved": kwork["flops"] / ksec / 1e12, "peak": tc_peak,
                "unit": "TFLOP/s", "peak_kind": "sustained" if sustained else "burst"}
    elif not tc_family and kwork["flops"] / 80e12 > kwork["bytes"] / (peaks["hbm_gbs"] * 1e9):
        # CUDA-core fp32 FMA: 152 SMs x 128 lanes x 2 flops x max SM clock
        alu_peak = 152 * 128 * 2 * peaks["sm_max_mhz"] * 1e6 / 1e12
        roof = {"bound": "alu", "achieved": kwork["flops"] / ksec / 1e12, "peak": alu_peak,
                "unit": "TFLOP/s", "peak_kind": "fp32 FMA at max SM clock"}
    else:
        roof = {"bound": "hbm", "achieved": kwork["bytes"] / ksec / 1e9, "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "peak_kind": "copy"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    return roof


def workload_name(cfg, T):
    return ("%s layer forward (d=%d f=%d E=%d top-%d shared %d), T=%d tokens, "
            "%d pool-resident / %d buffered experts"
            % (cfg.name, cfg.d, cfg.f, cfg.E, cfg.k, cfg.S * cfg.f, T, cfg.E - cfg.n_buffered,
               cfg.n_buffered))


def measure(lay, cfg_key, T, path_name, steps, warmup, device, dist, world, peaks, e2e=True):
    """One workload: K timed steps back to back (max over ranks), the dominant kernel bracketed
    by events in a second pass of K steps, and optionally K end-to-end steps with host copies."""
    pm, cfg = lay.pm, lay.cfg
    lay.plan.set_path(PATH_IDS[path_name])
    if lay.cplan is not None:
        lay.cplan.set_path(PATH_IDS[path_name])
    h_np, lg_np, hidden, logits = lay.tokens(T)
    e_act = lay.e_act(logits)
    wk = work(cfg, T, e_act)
    ws = pm.alloc_workspace(lay.desc, T, device)
    out = torch.empty_like(hidden)
    stream = torch.cuda.current_stream()

    def step():
        lay.plan.forward(hidden, logits, lay.page_table, lay.buf_slot, out=out, workspace=ws)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    path, nk, n_launch = lay.plan.last_run()
    assert lay.plan.device_error() == 0

    # which kernel dominates: one untimed pass with an event before every kernel
    probe = [torch.cuda.Event(enable_timing=True) for _ in range(nk + 1)]
    lay.plan.set_profile_events(probe)
    for _ in range(3):
        step()
    torch.cuda.synchronize()
    lay.plan.set_profile_events(None)
    probe_ms = [probe[j].elapsed_time(probe[j + 1]) for j in range(nk)]
    dom = int(np.argmax(probe_ms))

    # timed region: K steps back to back, with the dominant kernel bracketed by events on the
    # launching stream in every step (an event between two kernels keeps the second from starting
    # before the first ends, which costs the programmatic overlap at those two boundaries only)
    prof = []
    for _ in range(steps):
        evs = [None] * (nk + 1)
        evs[dom] = torch.cuda.Event(enable_timing=True)
        evs[dom + 1] = torch.cuda.Event(enable_timing=True)
        evs[dom].record(stream)        # created now, not inside the timed region
        evs[dom + 1].record(stream)
        prof.append(evs)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(steps):
        lay.plan.set_profile_events(prof[i])
        step()
    t_end.record(stream)
    torch.cuda.synchronize()
    lay.plan.set_profile_events(None)
    if dist:
        dist.barrier()
    region_s = t_start.elapsed_time(t_end) * 1e-3
    sec = max_over_ranks(region_s / steps, dist, device)
    dom_sec = float(np.mean([prof[i][dom].elapsed_time(prof[i][dom + 1]) for i in range(steps)])) * 1e-3
    assert lay.plan.device_error() == 0

    names = kernel_names(nk, path)
    kname = names[dom]
    wk["fused"] = {"flops": wk["flops"], "bytes": wk["bytes"]}
    roof = dominant_roofline(wk.get(kname, {"flops": 0.0, "bytes": 0.0}), dom_sec, path, peaks, region_s)
    roof["traffic"] = measured_traffic(cfg_key, T, PATH_NAMES[path], kname)
    roof["kernel"] = kname
    roof["kernel_ms"] = dom_sec * 1e3
    roof["peak_source"] = peaks["source"]
    res = {"cfg": cfg, "T": T, "path": path, "sec": sec, "region_s": region_s, "wk": wk,
           "e_act": e_act, "roofline": roof, "kernels_ms": {n: float(t) for n, t in zip(names, probe_ms)},
           "gpu_launches": int(n_launch * steps), "h_np": h_np, "lg_np": lg_np,
           "h2d": int(hidden.numel() * 2 + logits.numel() * 4), "d2h": int(out.numel() * 2)}
    if not e2e:
        return res

    # e2e: every step copies its inputs from pinned host memory and its result back, inside the
    # timed region.  Device buffers are double-buffered so step i+1's host->device copy and step
    # i-1's device->host copy (on their own streams) overlap step i's forward, ordered by events.
    h_host = hidden.cpu().pin_memory()
    l_host = logits.cpu().pin_memory()
    o_host = [torch.empty(out.shape, dtype=out.dtype, pin_memory=True) for _ in range(2)]
    hid_d = [hidden, torch.empty_like(hidden)]
    lg_d = [logits, torch.empty_like(logits)]
    out_d = [out, torch.empty_like(out)]
    cp_in, cp_out = torch.cuda.Stream(device=device), torch.cuda.Stream(device=device)
    in_ready = [torch.cuda.Event() for _ in range(2)]
    read_done = [torch.cuda.Event() for _ in range(2)]   # the forward of this slot finished
    out_done = [torch.cuda.Event() for _ in range(2)]    # the result of this slot is on the host
    for b in range(2):
        read_done[b].record(stream)
        out_done[b].record(stream)

    def e2e_step(i):
        b = i % 2
        with torch.cuda.stream(cp_in):
            cp_in.wait_event(read_done[b])           # the slot's previous forward has read it
            hid_d[b].copy_(h_host, non_blocking=True)
            lg_d[b].copy_(l_host, non_blocking=True)
            in_ready[b].record(cp_in)
        stream.wait_event(in_ready[b])
        stream.wait_event(out_done[b])               # the slot's previous result has left
        lay.plan.forward(hid_d[b], lg_d[b], lay.page_table, lay.buf_slot, out=out_d[b], workspace=ws)
        read_done[b].record(stream)
        with torch.cuda.stream(cp_out):
            cp_out.wait_event(read_done[b])
            o_host[b].copy_(out_d[b], non_blocking=True)
            out_done[b].record(cp_out)

    for i in range(3):
        e2e_step(i)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    cp_in.wait_event(e0)
    for i in range(steps):
        e2e_step(i)
    stream.wait_event(out_done[(steps - 1) % 2])   # the last result is on the host
    e1.record(stream)
    torch.cuda.synchronize()
    res["e2e_sec"] = max_over_ranks(e0.elapsed_time(e1) * 1e-3 / steps, dist, device)
    return res


CHAIN_LAYERS = 8
CHAIN_MAX_TOKENS = 32


def chain_plans(lay, n):
    """n more layers with the same weights and placement in page pools and load buffers of their
    own, so that a chain of distinct layers can be timed as a decode step runs it (each layer's
    pages streamed from HBM, the next layer's launch overlapping the previous one's tail)."""
    from paged_moe_expert_gb300 import pool as pl
    cfg, out = lay.cfg, []
    for _ in range(n):
        pool = pl.new_pool(cfg.num_pages, cfg.f, cfg.d, lay.device)
        bufs = pl.new_load_buffers(cfg.slots_per_buffer, cfg.f, cfg.d, lay.device)
        pt, bs = pl.place(cfg, lay.w, lay.placement, pool, bufs, 0)
        plan = lay.pm.Plan(lay.desc, pool, cfg.num_pages, bufs)
        out.append((plan, pool, bufs, pt.to(lay.device), bs.to(lay.device)))
    return out


def token_sweep(lay, iters, peaks, device):
    """Every token count of the workload: paged and contiguous forward replayed from CUDA graphs,
    interleaved, L2 flushed before every timed call (short bursts: the burst bf16 peak).  Decode
    sizes (up to 32 tokens) are also timed per layer in a chain of CHAIN_LAYERS distinct layers
    (one graph, L2 flushed before the chain), the way consecutive layers of a decode step run."""
    pm, cfg = lay.pm, lay.cfg
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=device)
    sweep = []
    lay.plan.set_path(pm.PATH_AUTO)
    lay.cplan.set_path(pm.PATH_AUTO)
    chain = chain_plans(lay, CHAIN_LAYERS) if min(cfg.tokens) <= CHAIN_MAX_TOKENS else []
    for Ts in cfg.tokens:
        _, _, hs, ls = lay.tokens(Ts)
        wss = pm.alloc_workspace(lay.desc, Ts, device)
        os_ = torch.empty_like(hs)
        fp = lambda: lay.plan.forward(hs, ls, lay.page_table, lay.buf_slot, out=os_, workspace=wss)  # noqa: E731
        fc = lambda: lay.cplan.contig_forward(hs, ls, out=os_, workspace=wss)  # noqa: E731
        for _ in range(3):
            fp(); fc()
        ps = lay.plan.last_run()[0]
        gp, gc = capture(fp), capture(fc)
        tp, tc = time_iters([gp.replay, gc.replay], iters, flush)
        # a timing is only a timing if no kernel reported an error (a bounded wait that ran
        # out would otherwise show up as a slow point)
        for pl_ in (lay.plan, lay.cplan):
            if pl_.device_error() != 0:
                raise RuntimeError("device error word set during the %d-token sweep point" % Ts)
        ea = lay.e_act(ls)
        wk_s = work(cfg, Ts, ea)
        frac, bound = binding_fraction(wk_s["flops"], wk_s["bytes"], tp, peaks, sustained=False)
        point = {"tokens": Ts, "path": PATH_NAMES[ps], "launch": "cuda_graph", "ms": tp * 1e3,
                 "contig_ms": tc * 1e3, "overhead_vs_contig": tp / tc - 1.0,
                 "tflops": wk_s["flops"] / tp / 1e12,
                 "weight_gbs": wk_s["weight_bytes"] / tp / 1e9,
                 "tokens_per_s": Ts / tp, "experts_active": ea,
                 "binding_roof": bound, "roof_frac": frac}
        if chain and Ts <= CHAIN_MAX_TOKENS:
            outs = [torch.empty_like(hs) for _ in chain]

            def run_chain():
                for (pln, _, _, pt_, bs_), o_ in zip(chain, outs):
                    pln.forward(hs, ls, pt_, bs_, out=o_, workspace=wss)
            run_chain()
            gch = capture(run_chain)
            tch, = time_iters([gch.replay], max(iters // 4, 5), flush)
            for pln, _, _, _, _ in chain:
                if pln.device_error() != 0:
                    raise RuntimeError("device error word set during the %d-token chain" % Ts)
            per = tch / len(chain)
            cfrac, _ = binding_fraction(wk_s["flops"], wk_s["bytes"], per, peaks, sustained=False)
            point.update({"chain_layers": len(chain), "chain_ms_per_layer": per * 1e3, "chain_roof_frac": cfrac})
            del gch, outs
        sweep.append(point)
        del wss, gp, gc
    del chain
    torch.cuda.empty_cache()
    return sweep


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="mixtral", choices=sorted(syn.CONFIGS))
    ap.add_argument("--tokens", type=int, default=0)
    ap.add_argument("--path", default="auto", choices=sorted(PATH_IDS))
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the other layer shapes (headline workload only)")
    ap.add_argument("--sweep-iters", type=int, default=50)
    ap.add_argument("--decode-sweep", action="store_true",
                    help="24-layer decode sweep with prefetch (prints one line per case)")
    ap.add_argument("--layers", type=int, default=24)
    ap.add_argument("--tokens-list", default="1,4,16,64,256")
    ap.add_argument("--fractions", default="1.0,0.875,0.75,0.625,0.5")
    ap.add_argument("--backend", default="host", choices=["host", "compressed"],
                    help="decode sweep: where offloaded experts live")
    ap.add_argument("--predicted", action="store_true",
                    help="decode sweep: prefetch from the previous step's routing and copy in "
                         "the experts it missed")
    ap.add_argument("--codec", action="store_true",
                    help="exponent-only Huffman decode of expert pages vs the host copy")
    ap.add_argument("--vmm-overhead", action="store_true",
                    help="page lookup vs remapped contiguous view vs contiguous allocation")
    ap.add_argument("--elastic-sweep", action="store_true",
                    help="adjuster-driven 24-layer decode over a KV demand trace")
    ap.add_argument("--elastic-requests", action="store_true",
                    help="elastic decode with request KV pages carved from the expert pool")
    ap.add_argument("--elastic-tokens", type=int, default=16)
    ap.add_argument("--offload-limit", type=int, default=30)
    ap.add_argument("--kv-peak", type=int, default=1800)
    args = ap.parse_args()
    if args.decode_sweep:
        decode_sweep(args)
        return
    if args.elastic_sweep:
        elastic_sweep(args)
        return
    if args.elastic_requests:
        elastic_requests(args)
        return
    if args.vmm_overhead:
        vmm_overhead(args)
        return
    if args.codec:
        codec_bench(args)
        return

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank)
        return
    if args.warmup < 3:
        args.warmup = 3

    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)

    peaks = load_peaks()
    cfg = syn.CONFIGS[args.config]
    T = args.tokens or cfg.tokens[-1]
    lay = Layer(cfg, device, contiguous=not args.no_sweep)

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    r = measure(lay, args.config, T, args.path, args.steps, args.warmup, device, dist, world, peaks)
    sweeps = {}
    if not args.no_sweep and rank == 0:
        sweeps[args.config] = token_sweep(lay, args.sweep_iters, peaks, device)
    clk = clocks.stop()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        cpu = oracle_throughput(cfg, lay.w, r["h_np"], r["lg_np"], 15.0, T)

    # the other layer shapes at their largest token count, and their token sweeps (rank 0 only)
    extra = []
    if not args.no_extra and rank == 0 and world == 1:
        del lay
        torch.cuda.empty_cache()
        for key in ("qwen15", "qwen3next"):
            if key == args.config:
                continue
            c2 = syn.CONFIGS[key]
            lay2 = Layer(c2, device, contiguous=not args.no_sweep)
            r2 = measure(lay2, key, c2.tokens[-1], "auto", args.steps, args.warmup, device, None, 1,
                         peaks, e2e=False)
            ov = None
            if not args.no_sweep:
                sweeps[key] = token_sweep(lay2, args.sweep_iters, peaks, device)
                ov = next((p["overhead_vs_contig"] for p in sweeps[key] if p["tokens"] == c2.tokens[-1]), None)
            extra.append({"workload": workload_name(c2, c2.tokens[-1]), "tokens": c2.tokens[-1],
                          "path": PATH_NAMES[r2["path"]], "tflops": r2["wk"]["flops"] / r2["sec"] / 1e12,
                          "ms_per_step": r2["sec"] * 1e3, "experts_active": r2["e_act"],
                          "weight_gbs": r2["wk"]["weight_bytes"] / r2["sec"] / 1e9,
                          "roofline": r2["roofline"], "kernels_ms": r2["kernels_ms"],
                          "overhead_vs_contig": ov})
            del lay2
            torch.cuda.empty_cache()

    sweep = sweeps.get(args.config, [])
    overhead = next((s_["overhead_vs_contig"] for s_ in sweep if s_["tokens"] == T), None)
    wk, sec = r["wk"], r["sec"]
    value = job_throughput(wk["flops"], world, sec) / 1e12
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": sec * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": workload_name(cfg, T),
                   "tokens": T, "path": PATH_NAMES[r["path"]], "experts_active": r["e_act"],
                   "weight_gbs": job_throughput(wk["weight_bytes"], world, sec) / 1e9,
                   "tokens_per_s": job_throughput(T, world, sec),
                   "l2": "inputs larger than L2 (%.0f MB of expert weights per step); sweeps flush L2"
                         % (wk["weight_bytes"] / 1e6),
                   "timed_region_s": r["region_s"],
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "roofline": r["roofline"],
        "cpu_baseline": cpu and {k: cpu[k] for k in ("value", "unit", "cores", "kind", "sample")},
        "e2e": {"value": job_throughput(wk["flops"], world, r["e2e_sec"]) / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"]},
        "gpu_launches": r["gpu_launches"],
        "clocks": clk,
        "kernels_ms": r["kernels_ms"],
        "overhead_vs_contig": overhead,
        "sweep": sweep,
        "extra_workloads": extra,
        "sweeps_other": {k: v for k, v in sweeps.items() if k != args.config},
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
