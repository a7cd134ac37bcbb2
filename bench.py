"""GPTQ per-layer benchmark on GB300 (one JSON line on rank 0).

A step is one pass of the whole layer path over one synthetic workload: the Hessian hook
over every calibration token, prepare (dead fix, act-order, damping, inverse Cholesky
factor) and the column loop with the lazy update, group scales/zeros, g_idx and packing.
The default workload is the q_proj-shaped layer (d_out = d_in = 4096, 128 x 2048 bf16
tokens, 4-bit asymmetric, group 128, act-order).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

With N > 1 (torchrun) every rank quantises its own replica of the layer (weak scaling,
no data-path collective); the step time is the maximum over ranks.  ``--impl
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
DEFAULT_CONFIG = "q_proj_4096x4096"
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


def source_hash(path: str) -> str:
    import hashlib
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


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

def run_ours(args, world, rank, local):
    import torch
    from post_weight_quantization_02_gb300 import LayerEngine, QuantizedLayer, gptq as G
    from post_weight_quantization_02_gb300 import quantize_layer_from_host
    from workloads import CONFIGS, channel_multipliers, make_tokens_chunk, make_weight

    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device (the engine has no CPU path)")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    dist = init_dist(world, "nccl")
    cfg = CONFIGS[args.config]
    if args.tokens:
        cfg = cfg.replace(n_tokens=args.tokens)
    m, d, n = cfg.d_out, cfg.d_in, cfg.n_tokens

    # synthetic workload, resident in HBM
    mult = channel_multipliers(cfg, dev)
    nch = -(-n // cfg.chunk)
    X = torch.cat([make_tokens_chunk(cfg, i, dev, mult) for i in range(nch)])
    W = make_weight(cfg, dev)
    eng = LayerEngine(m, d, cfg.bits, cfg.group, cfg.sym, cfg.actorder, cfg.damp,
                      cfg.blocksize, max_chunk_tokens=n, device=dev,
                      static_groups=args.static_groups)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        eng.reset()
        eng.add_batch(X)
        eng.prepare()
        eng.quantize_weights(W)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    # The timed steps trace the SYRK only (its CUDA-event duration is the roofline's
    # denominator); events around every kernel would cost time between the prepare's and
    # the quantize's kernels and break their dependent launches.
    G.gptq_profile_reset()
    G.gptq_profile_select([G.GPTQ_K_SYRK_TC])
    G.gptq_profile_enable(True)
    launches0 = G.gptq_launch_count()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    stops = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    with ClockSampler(dev.index) as clocks:
        barrier(dist, dev)
        torch.cuda.synchronize()
        wall0 = time.perf_counter()
        for i in range(args.steps):
            flush.fill_(float(i))              # evict L2 between steps (not timed)
            starts[i].record(stream)
            step()
            stops[i].record(stream)
        torch.cuda.synchronize()
        barrier(dist, dev)
        wall = time.perf_counter() - wall0
    G.gptq_profile_enable(False)
    launches = G.gptq_launch_count() - launches0
    step_ms = [a.elapsed_time(b) for a, b in zip(starts, stops)]
    ms_local = statistics.mean(step_ms)
    ms = max_over_ranks(dist, ms_local, dev)
    syrk_t, syrk_c = G.gptq_profile_read(G.GPTQ_K_SYRK_TC)

    # per-kernel breakdown: a separate, untimed pass with every kind traced
    kern = {}
    prof_steps = min(args.steps, 3)
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
        roofline = {"bound": "tensor", "kernel": "syrk_tc", "achieved": round(achieved, 1),
                    "peak": bf16, "unit": "TFLOP/s", "frac": round(achieved / bf16, 4),
                    "peak_source": f"{peak_src} bf16 dense burst",
                    # the measured power-capped figure (a GEMM run back to back), for context
                    "peak_sustained": bf16_sus,
                    "frac_of_sustained": round(achieved / bf16_sus, 4),
                    "algorithmic_flops_per_launch": flops,
                    "traffic": ncu_traffic("post_weight_quantization_02_gb300/csrc/hessian_tc.cu",
                                           args.config)}

    # end to end through the public API from pinned host memory
    e2e = None
    if not args.skip_e2e:
        e2e = run_e2e(args, cfg, X, W, eng, dist, dev, world)
    del X

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(cfg, None, W, budget_s=args.cpu_seconds)

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
            "kernels": {k: {kk: round(vv, 4) for kk, vv in v.items()} for k, v in kern.items()},
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def run_e2e(args, cfg, X, W, eng, dist, dev, world):
    """The same metric through the public API from pinned host buffers: host-to-device
    copies of every token chunk and of W, and the device-to-host copy of the packed
    outputs, are inside the timed region."""
    import torch
    from post_weight_quantization_02_gb300 import LayerEngine, QuantizedLayer
    from post_weight_quantization_02_gb300 import quantize_layer_from_host
    m, d, n = cfg.d_out, cfg.d_in, cfg.n_tokens
    Xh = X.cpu().pin_memory()
    Wh = W.cpu().pin_memory()
    chunk = cfg.chunk
    x_chunks = [Xh[i:i + chunk] for i in range(0, n, chunk)]
    out = QuantizedLayer(*(t.cpu().pin_memory() for t in
                           (eng.qweight, eng.scales, eng.qzeros, eng.g_idx, eng.perm, eng.loss)))
    e_eng = LayerEngine(m, d, cfg.bits, cfg.group, cfg.sym, cfg.actorder, cfg.damp,
                        cfg.blocksize, max_chunk_tokens=chunk, device=dev,
                        static_groups=args.static_groups)
    quantize_layer_from_host(e_eng, Wh, x_chunks, out)          # warm-up
    e_steps = max(1, min(args.steps, 5))
    barrier(dist, dev)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(e_steps):
        quantize_layer_from_host(e_eng, Wh, x_chunks, out)
    torch.cuda.synchronize()
    e_ms = max_over_ranks(dist, (time.perf_counter() - t0) * 1e3 / e_steps, dev)
    h2d = Xh.numel() * Xh.element_size() + Wh.numel() * Wh.element_size()
    d2h = sum(t.numel() * t.element_size() for t in
              (out.qweight, out.scales, out.qzeros, out.g_idx, out.perm, out.loss))
    return {"value": round(world * float(m) * d / (e_ms * 1e-3), 1), "unit": "weights/s",
            "ms_per_step": round(e_ms, 3), "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": e_steps,
            "path": f"quantize_layer_from_host, {len(x_chunks)} pinned chunks of {chunk} tokens"}


# ------------------------------------------------------------------------ CPU oracle

def oracle_layer_seconds(cfg, Xs, Ws, n_tokens_sample: int, rows_sample: int):
    """Time the float64 oracle on a bounded sample and extrapolate to the whole layer.

    Hessian on ``n_tokens_sample`` tokens (scaled by n / sample: the product is linear in
    tokens), the full prepare chain on the d_in x d_in matrix (not sampled), and the column
    loop on ``rows_sample`` output rows (scaled by d_out / rows: rows are independent).
    Returns (extrapolated seconds, measured seconds).
    """
    from oracle import gptq_oracle as O
    t0 = time.perf_counter()
    H = O.hessian(Xs[:n_tokens_sample])
    t1 = time.perf_counter()
    prep = O.gptq_prepare(H, cfg.damp, cfg.actorder)
    t2 = time.perf_counter()
    O.gptq_quantize_layer(Ws[:rows_sample], prep["U"], prep["perm"], prep["dead"], cfg.bits,
                          cfg.group, cfg.sym, cfg.blocksize, pack=False)
    t3 = time.perf_counter()
    full = ((t1 - t0) * cfg.n_tokens / n_tokens_sample + (t2 - t1)
            + (t3 - t2) * cfg.d_out / rows_sample)
    return full, t3 - t0


def cpu_sample_inputs(cfg, X=None, W=None, n_tokens_sample=4096):
    import numpy as np
    from workloads import make_tokens_chunk, make_weight
    if X is None:
        Xs = make_tokens_chunk(cfg, 0, "cpu")[:n_tokens_sample].float().numpy()
    else:
        Xs = X[:n_tokens_sample].float().cpu().numpy()
    Wm = make_weight(cfg, "cpu") if W is None else W
    return Xs.astype(np.float64), Wm.float().cpu().numpy().astype(np.float64)


def cpu_baseline(cfg, X=None, W=None, budget_s: float = 20.0):
    """The oracle as it stands, on this host's cores, on a bounded sample of the workload."""
    ntok, rows = 4096, 128
    Xs, Ws = cpu_sample_inputs(cfg, X, W, ntok)
    full, measured = oracle_layer_seconds(cfg, Xs, Ws, ntok, rows)
    return {"value": round(cfg.d_out * cfg.d_in / full, 1), "unit": "weights/s",
            "cores": os.cpu_count(), "kind": "oracle",
            "sample": (f"float64 numpy oracle: Hessian on {ntok} of {cfg.n_tokens} tokens "
                       f"(x{cfg.n_tokens // ntok}), full prepare on {cfg.d_in}^2, column loop "
                       f"on {rows} of {cfg.d_out} rows (x{cfg.d_out // rows}); "
                       f"{measured:.1f} s measured, {full:.1f} s extrapolated per layer"),
            "ms_per_layer_extrapolated": round(full * 1e3, 1)}


def run_reference(args, world, rank):
    """--impl reference: the float64 oracle, K timed steps of a bounded sample each."""
    if rank != 0:
        return
    from workloads import CONFIGS
    cfg = CONFIGS[args.config]
    ntok, rows = 2048, 64
    Xs, Ws = cpu_sample_inputs(cfg, n_tokens_sample=ntok)
    for _ in range(args.warmup):
        oracle_layer_seconds(cfg, Xs, Ws, ntok, rows)
    fulls, measured = [], 0.0
    for _ in range(args.steps):
        f, mt = oracle_layer_seconds(cfg, Xs, Ws, ntok, rows)
        fulls.append(f)
        measured += mt
    sec = statistics.mean(fulls)
    value = round(cfg.d_out * cfg.d_in / sec, 1)
    sample = (f"float64 numpy oracle per step: Hessian on {ntok} of {cfg.n_tokens} tokens, "
              f"full prepare on {cfg.d_in}^2, column loop on {rows} of {cfg.d_out} rows, "
              f"extrapolated to the whole layer")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "weights/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(sec * 1e3, 1), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
        "config": {"workload": cfg.name, "measured_cpu_s": round(measured, 2)},
        "cpu_baseline": {"value": value, "unit": "weights/s", "cores": os.cpu_count(),
                         "kind": "oracle", "sample": sample},
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
    """The block-sequential pipeline on a Llama-shaped block (hidden 4096, MLP 14336, 32
    heads, the 8B-class shapes of the survey's block configuration): Hessians of the four
    input groups over every calibration token, prepare, all seven linears quantised, and
    the re-forward with the dequantised weights.  One JSON line."""
    import torch
    from post_weight_quantization_02_gb300.pipeline import BlockQuantizer, make_block_weights

    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device (the engine has no CPU path)")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    dist = init_dist(world, "nccl")
    hidden, inter, heads, seq = 4096, 14336, 32, 2048
    tokens = args.tokens if args.tokens else 262144
    B = max(1, tokens // seq)
    g = torch.Generator(device="cpu").manual_seed(11)
    x = torch.randn(B, seq, hidden, generator=g).to(device=dev, dtype=torch.bfloat16)
    W = make_block_weights(hidden, inter, 1, dev)
    bq = BlockQuantizer(hidden, inter, heads, bits=4, group=128, static_groups=args.static_groups,
                        seqs_per_chunk=8, max_chunk_tokens=8 * seq, device=dev)
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
    weights = 4 * hidden * hidden + 3 * hidden * inter
    if rank == 0:
        print(json.dumps({
            "metric": "block-sequential GPTQ, ms per Llama-shaped block (and weights/s)",
            "value": round(ms, 3), "unit": "ms", "n_gpus": world, "steps": steps,
            "warmup": args.warmup, "higher_is_better": False, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (random-init block, seeded calibration tokens)",
            "config": {"workload": f"block hidden {hidden}, MLP {inter}, {heads} heads, "
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
                    help="timed steps (default: 100 for the layer path, about 0.6 s, so that "
                         "the clock sampler sees the timed region several times; 10 for "
                         "the other modes and the reference arm)")
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default=DEFAULT_CONFIG)
    ap.add_argument("--cpu-seconds", type=float, default=20.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--tokens", type=int, default=0,
                    help="override the calibration token count (small profiling cases)")
    ap.add_argument("--skip-e2e", action="store_true")
    ap.add_argument("--static-groups", action="store_true",
                    help="groups fixed in the original column order before the loop")
    ap.add_argument("--dequant-matmul", action="store_true",
                    help="measure the packed checkpoint's consumer instead of the layer path")
    ap.add_argument("--pipeline", action="store_true",
                    help="measure the block-sequential pipeline on a Llama-shaped block")
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)
    if args.steps is None:
        layer_path = not (args.impl == "reference" or args.dequant_matmul or args.pipeline)
        args.steps = 100 if layer_path else 10
    world, rank, local = dist_env()
    if args.impl == "reference":
        run_reference(args, world, rank)
    elif args.dequant_matmul:
        run_dequant(args, world, rank, local)
    elif args.pipeline:
        run_pipeline(args, world, rank, local)
    else:
        run_ours(args, world, rank, local)


if __name__ == "__main__":
    main()
