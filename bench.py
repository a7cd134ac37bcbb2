"""GPTQ per-layer benchmark on GB300 (one JSON line on rank 0).

A step is one pass of the whole layer path over one synthetic workload: the Hessian hook
over every calibration token, prepare (dead fix, act-order, damping, inverse Cholesky
factor) and the column loop with the lazy update, group scales/zeros, g_idx and packing.
The default workload is the 70B-width down_proj-shaped layer (d_out = 8192, d_in =
28672, 256 x 2048 bf16 tokens resident in HBM, 4-bit asymmetric, group 128, act-order),
the largest configuration that fits one GPU.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

With N > 1 (torchrun) every rank quantises its own replica of the layer (weak scaling,
no data-path collective); the step time is the maximum over ranks.  ``--shard`` splits
one layer across the ranks instead (strong scaling: token-sharded Hessian with one
all-reduce, replicated prepare, row-sharded quantize with one all-gather per output).  ``--impl
reference`` times the float64 CPU oracle on bounded samples of the same workload.
"""

from __future__ import annotations

import argparse
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

METRIC = "GPTQ per-layer time (ms) & weights/s at 4-bit g128; SYRK/GEMM TFLOP/s vs peak"
DEFAULT_CONFIG = "down_proj_8192x28672"
L2_FLUSH_BYTES = 256 << 20


# ------------------------------------------------------------------------ distributed

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world: int, backend: str):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)
    return dist if world > 1 else None


def barrier(dist, device=None):
    if dist is not None:
        if device is not None and device.type == "cuda":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def max_over_ranks(dist, value: float, device) -> float:
    """The largest of every rank's value (timing only; not part of the data path)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(dist, value: float, device) -> float:
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ------------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi samples (every 200 ms) of SM clock and throttle reasons while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, ValueError):
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
            if self.thread is not None:
                self.thread.join(timeout=2)

    def summary(self):
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for name, flag in zip(names, parts[4:8]):
                if flag.lower() in ("active", "1", "0x1"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------------ peaks, traffic

def measured_peaks():
    """(hbm GB/s, bf16 TFLOP/s burst, sustained, source) from MEASURED_PEAKS.json, else the
    recipe's fallback numbers."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), float(j["bf16_tflops"]), float(
            j.get("bf16_tflops_sustained", j["bf16_tflops"])), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, 1900.0, 1700.0, "fallback"


# the first line of the host-side part of the SYRK's source: the traffic figure depends
# on the device code above it, not on edits below it
HOST_PART_MARKER = "// CTAs' tiles per token split"


def source_hash(path: str) -> str:
    """Hash of a kernel file's device part (the text before HOST_PART_MARKER)."""
    import hashlib
    with open(path, "rb") as f:
        text = f.read()
    cut = text.find(HOST_PART_MARKER.encode())
    return hashlib.sha256(text if cut < 0 else text[:cut]).hexdigest()[:16]


def ncu_traffic(kernel_file: str, workload: str):
    """DRAM bytes per launch of the dominant kernel from the committed ncu summary, or
    None when the kernel source changed since the counters were taken."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            j = json.load(f)
        e = j[workload]
        if e["source_sha256_16"] != source_hash(os.path.join(ROOT, kernel_file)):
            return None
        return float(e["dram_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        return None


# ------------------------------------------------------------------------ our arm

def workload(args):
    """The configuration named by --config, with the --tokens / --shape overrides."""
    from workloads import CONFIGS
    cfg = CONFIGS[args.config]
    if getattr(args, "tokens", 0):
        cfg = cfg.replace(n_tokens=args.tokens)
    if getattr(args, "shape", None):
        cfg = cfg.replace(d_out=args.shape[0], d_in=args.shape[1])
    return cfg

BLOCK = 128  # the engine's column block


def algorithmic_work(cfg, n):
    """The algorithmic work of each step of the layer path (flops or bytes per layer)."""
    m, d = cfg.d_out, cfg.d_in
    we = 2 if "bfloat16" in str(cfg.w_dtype) else 4
    return {
        "syrk_flops": float(d) * (d + 1) * n,              # upper triangle of X^T X
        "cholesky_flops_pages": 4.0 * d ** 3 / 3,          # chol, cholesky_inverse, chol
        "cholesky_flops_engine": 2.0 * d ** 3 / 3,         # one factor + one triangular inverse
        "lazy_flops": float(m) * d * (d - BLOCK),          # sum over blocks of m x 128 x (d - i2)
        "loop_bytes": 13.0 * m * d,                        # W r/w, errors, codes
        "gather_bytes": float(m) * d * (we + 4),           # W in, permuted float32 copy out
        "pack_bytes": float(m) * d * (1 + cfg.bits / 8),   # codes in, packed words out
    }


def layer_figures(cfg, n, step_ms, phase_ms, kern, hbm, bf16, bf16_sus):
    """Achieved rates of each phase on its algorithmic work, as fractions of the measured
    peaks, and the step time against the sum of the kernels' roofline times."""
    w = algorithmic_work(cfg, n)

    def rate(x, ms, scale):
        return x / (ms * 1e-3) / scale if ms and ms > 0 else None

    def kms(name):
        k = kern.get(name)
        return k["ms_per_step"] if k else None

    def rnd(v, k=4):
        return None if v is None else round(v, k)

    prep_ms = phase_ms["prepare"]
    lazy_ms, loop_ms = kms("quant_lazy"), kms("quant_loop")
    gather_ms, pack_ms = kms("quant_gather"), kms("quant_pack")
    tp = rate(w["cholesky_flops_pages"], prep_ms, 1e12)
    te = rate(w["cholesky_flops_engine"], prep_ms, 1e12)
    tl = rate(w["lazy_flops"], lazy_ms, 1e12)
    gl = rate(w["loop_bytes"], loop_ms, 1e9)
    gg = rate(w["gather_bytes"], gather_ms, 1e9)
    gp = rate(w["pack_bytes"], pack_ms, 1e9)
    loop_launches = kern.get("quant_loop", {}).get("launches_per_step")
    figures = {
        "phases_ms": {k: round(v, 3) for k, v in phase_ms.items()},
        "prepare": {"ms": round(prep_ms, 3), "bound": "tensor (float32-accurate split products)",
                    "tflops_on_4d3_over_3": rnd(tp, 1), "tflops_on_2d3_over_3": rnd(te, 1),
                    "frac_of_bf16_burst": rnd(tp / bf16 if tp else None),
                    "frac_of_bf16_sustained": rnd(tp / bf16_sus if tp else None),
                    "note": "4d^3/3 is the pages' route (chol, inverse, chol); the engine's "
                            "route does 2d^3/3 (one factor, one triangular inverse)"},
        "lazy_update": {"kernel_ms": rnd(lazy_ms, 3), "bound": "tensor",
                        "algorithmic_flops": w["lazy_flops"], "tflops": rnd(tl, 1),
                        "frac_of_bf16_burst": rnd(tl / bf16 if tl else None),
                        "frac_of_bf16_sustained": rnd(tl / bf16_sus if tl else None)},
        "column_loop": {"kernel_ms": rnd(loop_ms, 3), "bound": "latency (column chain) / hbm",
                        "algorithmic_bytes": w["loop_bytes"], "gbs": rnd(gl, 1),
                        "frac_of_hbm": rnd(gl / hbm if gl else None),
                        "us_per_block": rnd(loop_ms * 1e3 / loop_launches
                                            if loop_ms and loop_launches else None, 2)},
        "gather": {"kernel_ms": rnd(gather_ms, 3), "bound": "hbm",
                   "algorithmic_bytes": w["gather_bytes"], "gbs": rnd(gg, 1),
                   "frac_of_hbm": rnd(gg / hbm if gg else None)},
        "pack": {"kernel_ms": rnd(pack_ms, 3), "bound": "hbm",
                 "algorithmic_bytes": w["pack_bytes"], "gbs": rnd(gp, 1),
                 "frac_of_hbm": rnd(gp / hbm if gp else None)},
    }
    # each kernel at its roofline (bf16 burst peak for the contractions, HBM for the rest)
    roof = {
        "syrk": w["syrk_flops"] / (bf16 * 1e12) * 1e3,
        "cholesky_chain": w["cholesky_flops_pages"] / (bf16 * 1e12) * 1e3,
        "lazy_update": w["lazy_flops"] / (bf16 * 1e12) * 1e3,
        "column_loop": w["loop_bytes"] / (hbm * 1e9) * 1e3,
        "gather": w["gather_bytes"] / (hbm * 1e9) * 1e3,
        "pack": w["pack_bytes"] / (hbm * 1e9) * 1e3,
    }
    total = sum(roof.values())
    figures["roofline_sum"] = {"ms": round(total, 3),
                               "per_kernel_ms": {k: round(v, 4) for k, v in roof.items()},
                               "step_frac_of_roofline_sum": round(total / step_ms, 4)}
    return figures


def run_ours(args, world, rank, local):
    import torch
    from post_weight_quantization_02_gb300 import LayerEngine, gptq as G
    from workloads import CONFIGS, channel_multipliers, make_tokens_chunk, make_weight

    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device (the engine has no CPU path)")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    dist = init_dist(world, "nccl")
    cfg = workload(args)
    m, d, n = cfg.d_out, cfg.d_in, cfg.n_tokens

    # synthetic workload, resident in HBM (chunks written straight into one tensor)
    mult = channel_multipliers(cfg, dev)
    X = torch.empty(n, d, dtype=cfg.x_dtype, device=dev)
    for i, t0 in enumerate(range(0, n, cfg.chunk)):
        X[t0:t0 + cfg.chunk] = make_tokens_chunk(cfg, i, dev, mult)
    W = make_weight(cfg, dev)
    eng = LayerEngine(m, d, cfg.bits, cfg.group, cfg.sym, cfg.actorder, cfg.damp,
                      cfg.blocksize, max_chunk_tokens=n, device=dev,
                      static_groups=args.static_groups)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        eng.reset()
        eng.add_batch(X)
        if ev is not None:
            ev[1].record(stream)
        eng.prepare()
        if ev is not None:
            ev[2].record(stream)
        eng.quantize_weights(W)
        if ev is not None:
            ev[3].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    # The timed steps trace the SYRK only (its CUDA-event duration is the roofline's
    # denominator); events around every kernel would cost time between the prepare's and
    # the quantize's kernels and break their dependent launches.  Four events per step,
    # between the three calls, give the phase times.
    G.gptq_profile_reset()
    G.gptq_profile_select([G.GPTQ_K_SYRK_TC])
    G.gptq_profile_enable(True)
    launches0 = G.gptq_launch_count()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    with ClockSampler(dev.index) as clocks:
        barrier(dist, dev)
        torch.cuda.synchronize()
        wall0 = time.perf_counter()
        for i in range(args.steps):
            flush.fill_(float(i))              # evict L2 between steps (not timed)
            step(evs[i])
        torch.cuda.synchronize()
        barrier(dist, dev)
        wall = time.perf_counter() - wall0
    G.gptq_profile_enable(False)
    launches = G.gptq_launch_count() - launches0
    step_ms = [e[0].elapsed_time(e[3]) for e in evs]
    phase_ms = {"hessian": statistics.mean(e[0].elapsed_time(e[1]) for e in evs),
                "prepare": statistics.mean(e[1].elapsed_time(e[2]) for e in evs),
                "quantize": statistics.mean(e[2].elapsed_time(e[3]) for e in evs)}
    ms_local = statistics.mean(step_ms)
    ms = max_over_ranks(dist, ms_local, dev)
    syrk_t, syrk_c = G.gptq_profile_read(G.GPTQ_K_SYRK_TC)

    # per-kernel breakdown: a separate, untimed pass with every kind traced
    kern = {}
    prof_steps = max(1, min(args.steps, 2))
    G.gptq_profile_reset()
    G.gptq_profile_select(None)
    G.gptq_profile_enable(True)
    for i in range(prof_steps):
        flush.fill_(float(i))
        step()
    torch.cuda.synchronize()
    G.gptq_profile_enable(False)
    for k in range(G.KERNEL_KINDS):
        t, c = G.gptq_profile_read(k)
        if c:
            kern[G.gptq_kernel_name(k)] = {"ms_per_step": t / prof_steps,
                                           "launches_per_step": c / prof_steps}

    hbm, bf16, bf16_sus, peak_src = measured_peaks()
    roofline = None
    if syrk_c:
        syrk_ms = syrk_t / syrk_c                       # live, over the timed steps
        flops = float(d) * (d + 1) * n                  # upper triangle of X^T X, 2 flop/MAC
        achieved = flops / (syrk_ms * 1e-3) / 1e12
        # The SYRK is timed inside a long run of steps (seconds of back-to-back work under
        # the power cap), so its roofline is the measured sustained bf16 figure; the burst
        # figure (a GEMM timed alone) is reported beside it.
        roofline = {"bound": "tensor", "kernel": "syrk_tc", "achieved": round(achieved, 1),
                    "peak": bf16_sus, "unit": "TFLOP/s", "frac": round(achieved / bf16_sus, 4),
                    "peak_source": f"{peak_src} bf16 dense sustained (GEMM back to back under "
                                   f"the power cap)",
                    "peak_burst": bf16,
                    "frac_of_burst": round(achieved / bf16, 4),
                    "ms_per_launch": round(syrk_ms, 3),
                    "algorithmic_flops_per_launch": flops,
                    "traffic": ncu_traffic("post_weight_quantization_02_gb300/csrc/hessian_tc.cu",
                                           cfg.name if not (args.tokens or args.shape) else None)}
    figures = layer_figures(cfg, n, ms, phase_ms, kern, hbm, bf16, bf16_sus)

    # end to end through the C ABI's host-buffer call
    e2e = None
    if not args.skip_e2e:
        e2e = run_e2e(args, cfg, X, W, eng, dist, dev, world)
    del X

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(cfg)

    total_launches = sum_over_ranks(dist, float(launches), dev)
    if rank == 0:
        weights = float(m) * d
        line = {
            "metric": METRIC,
            "value": round(world * weights / (ms * 1e-3), 1),
            "unit": "weights/s",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": round(ms, 4),
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "bf16",
            "data": "synthetic (seeded; shapes and distributions of the pages' workloads)",
            "config": {"workload": f"{cfg.name}: d_out={m} d_in={d}, {n} {str(cfg.x_dtype)[6:]} "
                                   f"calibration tokens, {cfg.bits}-bit "
                                   f"{'sym' if cfg.sym else 'asym'} group {cfg.group}, "
                                   f"act-order {'on' if cfg.actorder else 'off'}, damp {cfg.damp}"
                                   + (", static groups" if args.static_groups else ""),
                       "per_rank": "one independent layer replica per GPU",
                       "l2": "flushed between steps (256 MiB write, untimed); X > L2",
                       "step": "hessian_accumulate(all tokens) + prepare + quantize_layer",
                       "wall_s_timed_region": round(wall, 4)},
            "clocks": clocks.summary(),
            "e2e": e2e,
            "gpu_launches": int(total_launches),
            "roofline": roofline,
            "figures": figures,
            "kernels": {k: {kk: round(vv, 4) for kk, vv in v.items()} for k, v in kern.items()},
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def run_sharded(args, world, rank, local):
    """--shard: one layer split across the ranks (strong scaling): each rank runs the
    hook over its slice of the calibration tokens, the partial Hessians are rescaled and
    summed by one all-reduce, every rank prepares, each quantises its slice of rows, and
    one all-gather per output assembles the packed layer.  The step time is the maximum
    over ranks; ``value`` is the one layer's weights per second."""
    import torch
    from post_weight_quantization_02_gb300 import LayerEngine, ShardedLayer, shard
    from workloads import CONFIGS, channel_multipliers, make_tokens_chunk, make_weight

    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device (the engine has no CPU path)")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    dist = init_dist(world, "nccl")
    cfg = workload(args)
    m, d, n = cfg.d_out, cfg.d_in, cfg.n_tokens
    t0, t1 = shard.token_range(rank, world, n)
    r0, r1 = shard.row_range(rank, world, m)
    mult = channel_multipliers(cfg, dev)
    X = torch.empty(t1 - t0, d, dtype=cfg.x_dtype, device=dev)
    for i, c0 in enumerate(range(0, n, cfg.chunk)):
        a, b = max(c0, t0), min(c0 + cfg.chunk, t1)
        if a < b:
            X[a - t0:b - t0] = make_tokens_chunk(cfg, i, dev, mult)[a - c0:b - c0]
    W = make_weight(cfg, dev)[r0:r1].contiguous()
    eng = LayerEngine(r1 - r0, d, cfg.bits, cfg.group, cfg.sym, cfg.actorder, cfg.damp,
                      cfg.blocksize, max_chunk_tokens=max(1, t1 - t0), device=dev)
    sl = ShardedLayer(eng, m)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def step():
        sl.reset()
        sl.add_batch(X)
        sl.quantize(W)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    times = []
    with ClockSampler(dev.index) as clocks:
        for i in range(args.steps):
            flush.fill_(float(i))
            barrier(dist, dev)
            torch.cuda.synchronize()
            a = time.perf_counter()
            step()
            torch.cuda.synchronize()
            times.append(max_over_ranks(dist, (time.perf_counter() - a) * 1e3, dev))
    ms = statistics.mean(times)
    if rank == 0:
        print(json.dumps({
            "metric": METRIC, "value": round(float(m) * d / (ms * 1e-3), 1),
            "unit": "weights/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "strong",
            "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded; shapes and distributions of the pages' workloads)",
            "config": {"workload": f"{cfg.name}: d_out={m} d_in={d}, {n} tokens, one layer "
                                   f"split over {world} ranks",
                       "split": "tokens for the Hessian (rescale + all-reduce), prepare "
                                "replicated, rows for the quantize (all-gather)",
                       "l2": "flushed between steps (256 MiB write, untimed)",
                       "timing": "host wall clock per step, synchronised, max over ranks"},
            "clocks": clocks.summary(),
        }), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def run_e2e(args, cfg, X, W, eng, dist, dev, world):
    """The same metric through the C ABI's host-buffer call (gptq_quantize_layer_host):
    the host-to-device copies of every token chunk and of W, and the device-to-host copies
    of the packed outputs, are inside the timed region."""
    import torch
    from post_weight_quantization_02_gb300 import quantize_layer_from_host
    m, d, n = cfg.d_out, cfg.d_in, cfg.n_tokens
    Xh = torch.empty(X.shape, dtype=X.dtype, pin_memory=True)
    Xh.copy_(X)
    Wh = torch.empty(W.shape, dtype=W.dtype, pin_memory=True)
    Wh.copy_(W)
    out = quantize_layer_from_host(eng, Wh, Xh, chunk_tokens=cfg.chunk)   # warm-up
    # the host-to-device link's rate on this machine (untimed): one chunk copied 8 times
    stage = torch.empty(min(cfg.chunk, n), d, dtype=X.dtype, device=dev)
    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a0.record()
    for _ in range(8):
        stage.copy_(Xh[:stage.shape[0]], non_blocking=True)
    a1.record()
    torch.cuda.synchronize()
    link_gbs = 8 * stage.numel() * stage.element_size() / (a0.elapsed_time(a1) * 1e-3) / 1e9
    del stage
    e_steps = max(1, min(args.steps, 3))
    barrier(dist, dev)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(e_steps):
        quantize_layer_from_host(eng, Wh, Xh, out, chunk_tokens=cfg.chunk)
    torch.cuda.synchronize()
    e_ms = max_over_ranks(dist, (time.perf_counter() - t0) * 1e3 / e_steps, dev)
    h2d = Xh.numel() * Xh.element_size() + Wh.numel() * Wh.element_size()
    d2h = sum(t.numel() * t.element_size() for t in
              (out.qweight, out.scales, out.qzeros, out.g_idx, out.perm)) + 8
    del Xh, Wh
    return {"value": round(world * float(m) * d / (e_ms * 1e-3), 1), "unit": "weights/s",
            "ms_per_step": round(e_ms, 3), "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": e_steps,
            "h2d_link_gbs": round(link_gbs, 1),
            "h2d_copy_ms_at_link_rate": round(h2d / (link_gbs * 1e9) * 1e3, 1),
            "path": f"gptq_quantize_layer_host (C ABI): page-locked X copied in "
                    f"{-(-n // cfg.chunk)} chunks of {cfg.chunk} tokens overlapped with the "
                    f"Hessian kernels, then W; packed outputs copied back"}


# ------------------------------------------------------------------------ CPU oracle

def oracle_sample(cfg, ds: int = 4096, ms: int = 256, ns: int = 4096):
    """Time the float64 oracle, as it stands, on a bounded sample of the workload.

    The sample is the same workload scaled down: d_in' = min(d_in, ds) channels, d_out' =
    min(d_out, ms) rows and n' = min(n, ns) tokens drawn by the same generators.  Each
    phase is timed and scaled to the full layer by its operation count: the Hessian by
    (n/n') (d/d')^2, the prepare (dead fix, act-order, damping, inverse Cholesky factor) by
    (d/d')^3, the column loop and packing by (m/m') (d/d')^2.  Returns (seconds per layer
    extrapolated, seconds measured, description).
    """
    import numpy as np
    from oracle import gptq_oracle as O
    from workloads import make_tokens_chunk, make_weight
    sub = cfg.replace(d_in=min(ds, cfg.d_in), d_out=min(ms, cfg.d_out),
                      n_tokens=min(ns, cfg.n_tokens), chunk=min(ns, cfg.n_tokens))
    Xs = make_tokens_chunk(sub, 0, "cpu").float().numpy().astype(np.float64)
    Ws = make_weight(sub, "cpu").float().numpy().astype(np.float64)
    t0 = time.perf_counter()
    H = O.hessian(Xs)
    t1 = time.perf_counter()
    prep = O.gptq_prepare(H, sub.damp, sub.actorder)
    t2 = time.perf_counter()
    O.gptq_quantize_layer(Ws, prep["U"], prep["perm"], prep["dead"], sub.bits, sub.group,
                          sub.sym, sub.blocksize, pack=True)
    t3 = time.perf_counter()
    rd = cfg.d_in / sub.d_in
    full = ((t1 - t0) * (cfg.n_tokens / sub.n_tokens) * rd ** 2 + (t2 - t1) * rd ** 3
            + (t3 - t2) * (cfg.d_out / sub.d_out) * rd ** 2)
    exact = sub == cfg.replace(chunk=sub.chunk)
    desc = (f"float64 numpy oracle on a scaled-down copy of the workload: d_in {sub.d_in} of "
            f"{cfg.d_in}, d_out {sub.d_out} of {cfg.d_out}, {sub.n_tokens} of {cfg.n_tokens} "
            f"tokens, same generators and quantiser; " +
            ("the whole layer, not extrapolated" if exact else
             "phases scaled by their operation counts (Hessian n d^2, prepare d^3, column "
             "loop m d^2): extrapolated"))
    return full, t3 - t0, desc


def cpu_baseline(cfg):
    """The oracle as it stands, on this host's cores, on a bounded sample of the workload."""
    full, measured, desc = oracle_sample(cfg)
    return {"value": round(cfg.d_out * cfg.d_in / full, 1), "unit": "weights/s",
            "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{desc}; {measured:.2f} s measured, {full:.1f} s per layer",
            "ms_per_layer_extrapolated": round(full * 1e3, 1)}


def run_reference(args, world, rank):
    """--impl reference: the float64 oracle, K timed steps of a bounded sample each."""
    if rank != 0:
        return
    from workloads import CONFIGS
    cfg = workload(args)
    for _ in range(args.warmup):
        oracle_sample(cfg)
    fulls, walls = [], []
    desc = ""
    for _ in range(args.steps):
        f, mt, desc = oracle_sample(cfg)
        fulls.append(f)
        walls.append(mt)
    sec = statistics.mean(fulls)
    value = round(cfg.d_out * cfg.d_in / sec, 1)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "weights/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(statistics.mean(walls) * 1e3, 1),
        "ms_per_layer_extrapolated": round(sec * 1e3, 1),
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
        "config": {"workload": cfg.name,
                   "step": "one bounded sample of the workload through the oracle; "
                           "ms_per_step is the sample's measured time, value the layer "
                           "throughput extrapolated from it"},
        "cpu_baseline": {"value": value, "unit": "weights/s", "cores": os.cpu_count(),
                         "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": "weights/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_dequant(args, world, rank, local):
    """The packed checkpoint's consumer, y = x W_hat^T (gptq_dequant_matmul), on the layer
    of ``--config`` quantized by the library: one JSON line per token count.  HBM-bound:
    the algorithmic bytes are the packed weights, scales, zeros and g_idx plus x and y;
    L2 is flushed before every launch (the checkpoint is smaller than L2)."""
    import torch
    from post_weight_quantization_02_gb300 import gptq as G
    from workloads import CONFIGS, make_permutation, make_upper_factor, make_weight

    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device (the engine has no CPU path)")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    dist = init_dist(world, "nccl")
    cfg = CONFIGS[args.config]
    m, d, bits = cfg.d_out, cfg.d_in, cfg.bits
    Gn = 1 if cfg.group == -1 else -(-d // cfg.group)
    W = make_weight(cfg, dev)
    U = make_upper_factor(d, cfg.seed, dev)
    perm = make_permutation(d, cfg.seed, dev)
    qw = torch.empty(bits * d // 32, m, dtype=torch.int32, device=dev)
    sc = torch.empty(Gn, m, dtype=torch.float32, device=dev)
    qz = torch.empty(Gn, bits * m // 32, dtype=torch.int32, device=dev)
    gi = torch.empty(d, dtype=torch.int32, device=dev)
    loss = torch.empty((), dtype=torch.float64, device=dev)
    G.gptq_quantize_layer(W, U, perm, None, bits, cfg.group, cfg.sym, cfg.blocksize, qw, sc, qz,
                          gi, loss, static_groups=args.static_groups)
    del W, U
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    ws = G.workspace(G.gptq_workspace_size(G.GPTQ_OP_DEQUANT_MATMUL, 0, m, d, bits, -1), dev)
    stream = torch.cuda.current_stream(dev)
    hbm, _, _, peak_src = measured_peaks()
    ckpt_bytes = (qw.numel() + qz.numel() + gi.numel()) * 4 + sc.numel() * 4
    for n in (1, 8, 16):
        x = torch.randn(n, d, device=dev).to(torch.bfloat16)
        y = torch.empty(n, m, dtype=torch.float32, device=dev)
        for _ in range(args.warmup):
            G.gptq_dequant_matmul(x, qw, sc, qz, gi, bits, y, ws)
        torch.cuda.synchronize()
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        stops = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        # the kernel's own CUDA-event time (library tracing of this kind only) and the
        # whole call's (status word cleared and read back, stream synchronised)
        G.gptq_profile_reset()
        G.gptq_profile_select([G.GPTQ_K_DEQUANT_MATMUL])
        G.gptq_profile_enable(True)
        with ClockSampler(dev.index) as clocks:
            barrier(dist, dev)
            for i in range(args.steps):
                flush.fill_(float(i))          # cold L2 for every launch (not timed)
                starts[i].record(stream)
                G.gptq_dequant_matmul(x, qw, sc, qz, gi, bits, y, ws)
                stops[i].record(stream)
            torch.cuda.synchronize()
            barrier(dist, dev)
        G.gptq_profile_enable(False)
        G.gptq_profile_select(None)
        kt, kc = G.gptq_profile_read(G.GPTQ_K_DEQUANT_MATMUL)
        us = max_over_ranks(dist, kt / max(kc, 1) * 1e3, dev)
        call_us = max_over_ranks(dist, statistics.mean(a.elapsed_time(b) for a, b in
                                                        zip(starts, stops)) * 1e3, dev)
        nbytes = ckpt_bytes + x.numel() * 2 + y.numel() * 4
        gbs = nbytes / (us * 1e-6) / 1e9
        if rank == 0:
            print(json.dumps({
                "metric": "dequant-matmul of the packed checkpoint (us per launch)",
                "value": round(us, 3), "unit": "us", "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "higher_is_better": False, "scaling": "weak",
                "vs_baseline": None, "dtype": "bf16 x, int codes, f32 accumulate",
                "data": "synthetic (the library's own checkpoint of a seeded layer)",
                "config": {"workload": f"{cfg.name}: y[{n}, {m}] = x[{n}, {d}] W_hat^T, "
                                       f"{bits}-bit group {cfg.group}"
                                       + (" static groups" if args.static_groups else
                                          " act-order groups"),
                           "l2": "flushed before every launch",
                           "call_us": round(call_us, 3)},
                "clocks": clocks.summary(),
                "roofline": {"bound": "hbm", "kernel": "dequant_matmul", "achieved": round(gbs, 1),
                             "peak": hbm, "unit": "GB/s", "frac": round(gbs / hbm, 4),
                             "peak_source": f"{peak_src} HBM copy",
                             "algorithmic_bytes_per_launch": nbytes, "traffic": None},
            }), flush=True)


def run_pipeline(args, world, rank, local):
    """The block-sequential pipeline on a Llama-3-8B-shaped block (hidden 4096, MLP 14336,
    32 query heads, 8 key/value heads: k and v are 1024 x 4096): Hessians of the four
    input groups over every calibration token, prepare, all seven linears quantised, and
    the re-forward with the dequantised weights.  One JSON line."""
    import torch
    from post_weight_quantization_02_gb300.pipeline import BlockQuantizer, make_block_weights

    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device (the engine has no CPU path)")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    dist = init_dist(world, "nccl")
    hidden, inter, heads, kv_heads, seq = 4096, 14336, 32, 8, 2048
    kv_dim = hidden * kv_heads // heads
    tokens = args.tokens if args.tokens else 262144
    B = max(1, tokens // seq)
    g = torch.Generator(device="cpu").manual_seed(11)
    x = torch.randn(B, seq, hidden, generator=g).to(device=dev, dtype=torch.bfloat16)
    W = make_block_weights(hidden, inter, 1, dev, kv_dim=kv_dim)
    bq = BlockQuantizer(hidden, inter, heads, bits=4, group=128, static_groups=args.static_groups,
                        seqs_per_chunk=8, max_chunk_tokens=8 * seq, device=dev,
                        kv_heads=kv_heads)
    for _ in range(max(1, args.warmup - 2)):
        bq.quantize_block(x, W)
    torch.cuda.synchronize()
    steps = max(1, min(args.steps, 5))
    with ClockSampler(dev.index) as clocks:
        barrier(dist, dev)
        t0 = time.perf_counter()
        for _ in range(steps):
            bq.quantize_block(x, W)
        torch.cuda.synchronize()
        barrier(dist, dev)
        ms = max_over_ranks(dist, (time.perf_counter() - t0) * 1e3 / steps, dev)
    weights = 2 * hidden * hidden + 2 * kv_dim * hidden + 3 * hidden * inter
    if rank == 0:
        print(json.dumps({
            "metric": "block-sequential GPTQ, ms per Llama-shaped block (and weights/s)",
            "value": round(ms, 3), "unit": "ms", "n_gpus": world, "steps": steps,
            "warmup": args.warmup, "higher_is_better": False, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (random-init block, seeded calibration tokens)",
            "config": {"workload": f"block hidden {hidden}, MLP {inter}, {heads} heads "
                                   f"({kv_heads} key/value heads), "
                                   f"{B * seq} tokens ({B} x {seq}), 4-bit group 128, act-order"
                                   + (", static groups" if args.static_groups else ""),
                       "step": "forward (4 Hessian groups) + 4 prepares + 7 quantisations "
                               "+ re-forward with the dequantised weights",
                       "weights_per_s": round(weights / (ms * 1e-3), 1)},
            "clocks": clocks.summary(),
        }), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default: 20 for the layer path, about 11 s on the "
                         "default workload, so that the clock sampler sees the timed region "
                         "many times; 10 for the other modes and the reference arm)")
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default=DEFAULT_CONFIG)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--tokens", type=int, default=0,
                    help="override the calibration token count (small profiling cases)")
    ap.add_argument("--shape", type=int, nargs=2, metavar=("D_OUT", "D_IN"), default=None,
                    help="override the layer shape (small profiling cases)")
    ap.add_argument("--skip-e2e", action="store_true")
    ap.add_argument("--static-groups", action="store_true",
                    help="groups fixed in the original column order before the loop")
    ap.add_argument("--shard", action="store_true",
                    help="split one layer across the ranks (tokens for the Hessian, rows "
                         "for the quantize) instead of one replica per rank")
    ap.add_argument("--dequant-matmul", action="store_true",
                    help="measure the packed checkpoint's consumer instead of the layer path")
    ap.add_argument("--pipeline", action="store_true",
                    help="measure the block-sequential pipeline on a Llama-shaped block")
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)
    if args.steps is None:
        layer_path = not (args.impl == "reference" or args.dequant_matmul or args.pipeline
                          or args.shard)
        args.steps = 20 if layer_path else 10
    world, rank, local = dist_env()
    if args.impl == "reference":
        run_reference(args, world, rank)
    elif args.dequant_matmul:
        run_dequant(args, world, rank, local)
    elif args.pipeline:
        run_pipeline(args, world, rank, local)
    elif args.shard:
        run_sharded(args, world, rank, local)
    else:
        run_ours(args, world, rank, local)


if __name__ == "__main__":
    main()
