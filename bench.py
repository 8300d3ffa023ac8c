"""Benchmark of the multi-head attention forward on GB300.

python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]
                [--pass fwd|bwd] [--eager] [--no-cpu-baseline]

One step = one mha_fwd call over the whole workload (every sequence, head and
query tile), inputs resident in HBM.  Prints ONE JSON line (rank 0).

Timing: after W warm-up steps the K timed steps' C-ABI calls are captured once
into a CUDA graph, which is replayed once untimed and once between CUDA events
on the launching stream (barrier + synchronize on both sides), so the device
runs the launches back to back; ``--eager`` issues them one by one with events
around each instead.  Consecutive steps rotate over enough input copies that
no step finds its inputs in L2.

Metric: attention forward TFLOP/s, FLOPs = 4*B*H*Lq*Lk*d_k (halved under the
causal mask), bf16 inputs, float32 accumulation; also reported as a fraction
of the measured dense bf16 tensor peak.  The roofline fraction counts the
(query, visible key) pairs (L(L+1)/2 per head under the causal mask, the drawn
key lengths under key padding), reported beside as ``value_algorithmic``.

The default forward run also times every configuration of the target
specification and the supplementary d_k = 64, L >= 2048 shapes (``configs``:
TFLOP/s, fraction of the tensor peak, GB/s of algorithmic bytes and fraction of
the HBM bandwidth, and the oracle's rate on all host cores and, for the three
smallest, on one core); ``--no-sweep`` skips it.  The default workload is the GPT-3-like
causal self-attention (B 4, H 96, d_k 128, L 2048): the only L >= 2048 shape of
the five the pages suggest, and the one the throughput target is quoted on.

N > 1 (torchrun, one rank per GPU): weak scaling; every rank runs its own
replica of the workload (rank-specific seed), no data-path collective.
``--impl reference`` times the float64 CPU oracle on the host cores on a
bounded sample of the same workload (rank 0 only).

``--pass bwd``: one step = one mha_bwd call (the gradient dq, dk, dv of the
workload for a seeded dout, with the forward's output and row lse resident);
FLOPs = 2.5x the forward's (five products over the visible pairs).

``--pass gemm``: the layers' projection GEMM (mha_gemm_bf16) alone, on the
GPT-3-like and base-model projection shapes, beside torch.matmul (cuBLAS) on
the same operands.

Decode workloads (``--workload gpt3_decode`` / ``base_decode`` /
``gpt3_decode_b1``): one step = one mha_decode call (every sequence's new
query against its key/value cache); the metric is the step's algorithmic
bytes (q, out, and the visible K and V rows) per second, against the measured
HBM bandwidth.
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

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from transformer_head_scaled_sdpa_gb300 import dist as mdist  # noqa: E402
from transformer_head_scaled_sdpa_gb300 import inputs  # noqa: E402

METRIC = "attention fwd TFLOP/s (bf16, 1 GB300) and % of dense BF16 tensor peak"
UNIT = "TFLOP/s"
PEAKS_PATH = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_BYTES = 129 * 1024 * 1024


def load_peaks():
    try:
        with open(PEAKS_PATH) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


F32_ALU_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12


def visible_pairs(w, key_lens) -> float:
    """(query, visible key) pairs: the algorithmic work unit."""
    if w.mask_kind == inputs.MASK_CAUSAL:
        L = w.Lq
        return w.B * w.H * L * (L + 1) / 2
    if w.mask_kind == inputs.MASK_CAUSAL_KEY_PADDING:
        # row i of sequence b sees min(i + 1, len_b) keys
        i = torch.arange(w.Lq, dtype=torch.int64)
        lens = key_lens.clamp(0, w.Lk).to(torch.int64)
        return float(w.H * torch.minimum(i[None, :] + 1, lens[:, None]).sum().item())
    if w.mask_kind == inputs.MASK_KEY_PADDING:
        lens = key_lens.clamp(0, w.Lk).to(torch.int64).sum().item()
        return w.H * w.Lq * float(lens)
    return float(w.B * w.H * w.Lq * w.Lk)


def workload_config(w, extra=None):
    cfg = {"workload": w.name, "B": w.B, "H": w.H, "Lq": w.Lq, "Lk": w.Lk, "d_k": w.d_k,
           "mask": inputs.MASK_NAMES[w.mask_kind], "input_scale": w.input_scale,
           "seed": w.seed, "layout": "[B, L, H, d_k]"}
    if extra:
        cfg.update(extra)
    return cfg


# ---------------------------------------------------------------------------
# clocks: nvidia-smi sampled during the timed region
# ---------------------------------------------------------------------------
def gpu_id(dev) -> str:
    """nvidia-smi --id of this device (its UUID: independent of CUDA_VISIBLE_DEVICES)."""
    uuid = str(getattr(torch.cuda.get_device_properties(dev), "uuid", "") or "")
    if uuid:
        return uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    return str(dev.index)


class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu: str):
        self.gpu = gpu
        self.proc = None
        self.lines = []
        self.marks = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, name):
        self.marks.append((name, time.time()))

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            self.proc.wait(5)
        except subprocess.TimeoutExpired:
            self.proc.kill()

    def summary(self, t0, t1):
        rows = []
        for ts, line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((ts, float(parts[1]), float(parts[2]), parts))
            except ValueError:
                continue
        inside = [r for r in rows if t0 <= r[0] <= t1]
        used = inside if inside else rows
        if not used:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in used:
            for name, val in zip(names, r[3][5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r[1] for r in used),
                "sm_max_mhz": max(r[2] for r in used),
                "reasons": sorted(reasons),
                "samples": len(used),
                "samples_in_timed_region": len(inside)}


def timed_steps(step, args, dev, stream, rank, warm=True):
    """args.steps steps between a barrier + synchronize on both sides (after
    args.warmup untimed ones when ``warm``), clocks sampled meanwhile.

    By default the steps are captured once into a CUDA graph (each step's
    launches, through the same C-ABI calls) and the graph is replayed once
    untimed and once timed, so the device runs the launches back to back and
    the host's per-call argument marshalling (tens of microseconds of Python)
    is not on the clock; the mean time per step is then the graph's time over
    args.steps.  With ``--eager`` the steps are issued one by one with CUDA
    events around each.  Returns (mean ms per step, total ms max over ranks,
    clock summary or None)."""
    if warm:
        with torch.cuda.stream(stream):
            for _ in range(args.warmup):
                step()
    torch.cuda.synchronize(dev)
    graph = None
    if not args.eager:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream, capture_error_mode="thread_local"):
            for _ in range(args.steps):
                step()
        with torch.cuda.stream(stream):
            graph.replay()
        torch.cuda.synchronize(dev)
    sampler = ClockSampler(gpu_id(dev))
    if rank == 0:
        sampler.start()
        time.sleep(0.3)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps if graph is None else 0)]
    all_start = torch.cuda.Event(enable_timing=True)
    all_end = torch.cuda.Event(enable_timing=True)
    mdist.barrier(dev)
    torch.cuda.synchronize(dev)
    t_wall0 = time.time()
    with torch.cuda.stream(stream):
        all_start.record(stream)
        if graph is not None:
            graph.replay()
        else:
            for i in range(args.steps):
                ev[i][0].record(stream)
                step()
                ev[i][1].record(stream)
        all_end.record(stream)
    torch.cuda.synchronize(dev)
    mdist.barrier(dev)
    t_wall1 = time.time()
    total_ms = all_start.elapsed_time(all_end)
    step_ms = (total_ms if graph is not None else sum(a.elapsed_time(b) for a, b in ev)) / args.steps
    max_total_ms = mdist.max_over_ranks(total_ms, dev)
    if rank == 0:
        time.sleep(0.3)
        sampler.stop()
    del graph
    return step_ms, max_total_ms, (sampler.summary(t_wall0, t_wall1) if rank == 0 else None)


def timing_config(args):
    return ({"timing": "eager: one C-ABI call per step, CUDA events around each"} if args.eager
            else {"timing": "CUDA graph of the steps' C-ABI launches, replayed once timed"})


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def traffic_record(kernel_fp: str, workload: str, kernel: str = "fwd_bf16_kernel"):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel source (null otherwise)."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    if rec.get("kernel_source_sha256") != kernel_fp:
        return None
    return rec.get("dram_bytes_per_launch")


# the sources each profiled kernel is compiled from
KERNEL_SOURCES = {
    "fwd_bf16_kernel": ("kernels.h", "mha_fwd_bf16.cu", "ptx.cuh"),
    "decode_split_kernel": ("kernels.h", "mha_decode.cu", "ptx.cuh"),
    "bwd_dkdv_kernel": ("kernels.h", "mha_bwd.cu", "ptx.cuh"),
}


def kernel_fingerprint(kernel: str = "fwd_bf16_kernel") -> str:
    """sha256 over the source files the kernel is compiled from."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "transformer_head_scaled_sdpa_gb300", "csrc")
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()


def cpu_baseline(w, case, budget_s=12.0, threads=None, min_s=0.0):
    """The oracle, as it stands, on a bounded sample of whole heads of the
    workload (cycling over the heads again while less than ``min_s`` seconds
    have passed, for workloads that take microseconds); returns TFLOP/s of
    algorithmic work and the sample description.  ``threads`` None: every
    core the process may use."""
    import oracle
    cores = oracle.default_threads() if threads is None else threads
    done_pairs = 0.0
    heads = 0
    t0 = time.perf_counter()
    b_h = [(b, h) for b in range(w.B) for h in range(w.H)]
    one = inputs.Workload(w.name, 1, 1, w.d_k, w.Lq, w.Lk, w.mask_kind, w.dtype)
    while heads < len(b_h) or time.perf_counter() - t0 < min_s:
        b, h = b_h[heads % len(b_h)]
        sub = {n: case[n][b:b + 1, :, h:h + 1] for n in ("q", "k", "v")}
        lens = case["key_lens"][b:b + 1] if case["key_lens"] is not None else None
        oracle.mha(sub["q"], sub["k"], sub["v"], w.mask_kind,
                   key_lens=lens.numpy() if lens is not None else None, threads=threads)
        heads += 1
        done_pairs += visible_pairs(one, lens)
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    flops = 4.0 * w.d_k * done_pairs
    return {"value": flops / dt / 1e12, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{heads} whole (b, h) heads of {w.name} ({w.Lq}x{w.Lk}, d_k {w.d_k}, "
                      f"{inputs.MASK_NAMES[w.mask_kind]}) in float64, {dt:.2f} s wall",
            "seconds": dt, "seconds_per_step": dt * w.B * w.H / heads}


def forward_sets(w, case, dev):
    """The workload's inputs on the device, rotated over enough copies that
    consecutive steps never find their inputs in L2 (when one set fits)."""
    q, k, v = (case[n].to(dev) for n in ("q", "k", "v"))
    out = torch.empty_like(q)
    bytes_in = sum(t.numel() * t.element_size() for t in (q, k, v))
    n_sets = 1 if bytes_in > L2_BYTES else -(-2 * L2_BYTES // bytes_in)
    sets = [(q, k, v, out)] + [tuple(t.clone() for t in (q, k, v, out))
                              for _ in range(n_sets - 1)]
    return sets, bytes_in


def fwd_kernel_label(w):
    """The forward kernel of the library's last launch (call it right after
    the workload's own launches): the float32 kernel for float32 workloads;
    for bf16 the one-tile kernel (heads wider than 128; short sequences of
    heads up to 64 wide) runs 256-thread CTAs, the two-tile kernel 384."""
    from transformer_head_scaled_sdpa_gb300 import binding
    if w.dtype != torch.bfloat16:
        return "fwd_f32_kernel"
    return "fwd_wide_kernel" if binding.last_launch_info()["block"] == 256 else "fwd_bf16_kernel"


def measure_forward(w, case, args, dev, stream, rank, steps, warmup):
    """Time `steps` forward calls of the workload (after `warmup`), inputs
    resident; returns (kernel ms per step, max-over-ranks total ms, clocks,
    launches per step, input bytes, sets rotated)."""
    from transformer_head_scaled_sdpa_gb300 import binding
    lens = case["key_lens"].to(dev) if case["key_lens"] is not None else None
    sets, bytes_in = forward_sets(w, case, dev)
    cur = [0]
    fwd = binding.mha_fwd if w.dtype == torch.bfloat16 else binding.mha_fwd_f32

    def step():
        qq, kk, vv, oo = sets[cur[0] % len(sets)]
        cur[0] += 1
        fwd(qq, kk, vv, out=oo, mask_kind=w.mask_kind, key_lens=lens, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(warmup):
            step()
    rc = binding.mha_sync_status(stream)
    if rc != 0:
        raise binding.MhaError(rc, f"warm-up of {w.name}")
    launches = binding.last_launch_info()["kernels"]
    timing = argparse.Namespace(steps=steps, warmup=0, eager=args.eager)
    kernel_ms, max_total_ms, clocks = timed_steps(step, timing, dev, stream, rank, warm=False)
    rc = binding.mha_sync_status(stream)
    if rc != 0:
        raise binding.MhaError(rc, f"timed region of {w.name}")
    del sets
    return kernel_ms, max_total_ms, clocks, launches, bytes_in


def host_link(dev, stream, nbytes=256 << 20, reps=3):
    """Pinned host <-> device copy bandwidth (GB/s): each direction alone and
    both at once (two streams), best of `reps`; the ceiling of the e2e path."""
    h_src = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    h_dst = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    d_a = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    d_b = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    other = torch.cuda.Stream(device=dev)

    def best(fn):
        t = []
        for _ in range(reps):
            torch.cuda.synchronize(dev)
            t0 = time.perf_counter()
            fn()
            torch.cuda.synchronize(dev)
            t.append(time.perf_counter() - t0)
        return min(t)

    def h2d():
        with torch.cuda.stream(stream):
            d_a.copy_(h_src, non_blocking=True)

    def d2h():
        with torch.cuda.stream(stream):
            h_dst.copy_(d_b, non_blocking=True)

    def both():
        with torch.cuda.stream(stream):
            d_a.copy_(h_src, non_blocking=True)
        with torch.cuda.stream(other):
            h_dst.copy_(d_b, non_blocking=True)

    h2d()
    d2h()
    r = {"h2d_gbs": nbytes / best(h2d) / 1e9, "d2h_gbs": nbytes / best(d2h) / 1e9,
         "both_gbs": 2 * nbytes / best(both) / 1e9, "bytes": nbytes,
         "how": "pinned torch copies on two streams, wall clock after synchronize, best of 3"}
    del h_src, h_dst, d_a, d_b
    return r


# Every configuration of the target specification plus the supplementary
# d_k = 64, L >= 2048 shapes and the head-width-256 shapes, with and without
# the causal mask: the default run times each one (the headline workload is
# measured once, above).
SWEEP = ["toy_cross_f32", "base_encoder_self", "base_decoder_causal", "base_cross_keypad",
         "gpt3_causal", "big16_L2048", "big16_L2048_causal", "base8_L4096",
         "base8_L4096_causal", "d256_L2048", "d256_L2048_causal"]
# the configurations whose oracle is also timed on a single core
ONE_CORE = {"toy_cross_f32", "base_encoder_self", "base_decoder_causal"}


def config_record(w, case, kernel_ms, launches, peaks, with_oracle, kernel):
    """One sweep row: nominal and algorithmic TFLOP/s, fractions of the
    measured tensor and HBM peaks, and the oracle's rate on the host cores."""
    pairs = visible_pairs(w, case["key_lens"])
    flops_alg = 4.0 * w.d_k * pairs
    flops_nom = w.flops()
    elem = 2 if w.dtype == torch.bfloat16 else 4
    # Q and O once, K and V once over the keys any query sees
    if w.mask_kind & inputs.MASK_KEY_PADDING:
        kv_rows = float(case["key_lens"].clamp(0, w.Lk).sum().item())
    else:
        kv_rows = float(w.B * w.Lk)
    bytes_alg = elem * w.H * w.d_k * (2.0 * w.B * w.Lq + 2.0 * kv_rows)
    tensor_peak = float(peaks["bf16_tflops"])
    hbm = float(peaks["hbm_gbs"])
    sec = kernel_ms * 1e-3
    rec = {"workload": w.name, "B": w.B, "H": w.H, "Lq": w.Lq, "Lk": w.Lk, "d_k": w.d_k,
           "mask": inputs.MASK_NAMES[w.mask_kind],
           "dtype": "bf16" if w.dtype == torch.bfloat16 else "f32",
           "us_per_step": kernel_ms * 1e3, "launches_per_step": launches,
           "kernel": kernel,
           "tflops": flops_nom / sec / 1e12,
           "tflops_algorithmic": flops_alg / sec / 1e12,
           "frac_tensor_peak": (flops_alg / sec / 1e12 / tensor_peak
                                if w.dtype == torch.bfloat16 else None),
           "gbs": bytes_alg / sec / 1e9, "frac_hbm": bytes_alg / sec / 1e9 / hbm,
           "algorithmic_bytes": bytes_alg,
           "bound": ("alu" if w.dtype != torch.bfloat16 else
                     "tensor" if flops_alg / bytes_alg > tensor_peak * 1e3 / hbm else "hbm")}
    if w.dtype != torch.bfloat16:
        rec["frac_alu_peak"] = flops_alg / sec / 1e12 / F32_ALU_TFLOPS
    if with_oracle:
        o = cpu_baseline(w, case, budget_s=2.0, min_s=0.5)
        rec["oracle_all_cores"] = {k: o[k] for k in ("value", "unit", "cores", "sample",
                                                     "seconds_per_step")}
        if w.name in ONE_CORE:
            o1 = cpu_baseline(w, case, budget_s=2.0, threads=1, min_s=0.5)
            rec["oracle_one_core"] = {k: o1[k] for k in ("value", "unit", "cores", "sample",
                                                         "seconds_per_step")}
    return rec


def run_ours(args):
    rank, world = mdist.init("nccl")
    _, _, local_rank = mdist.env_rank_world()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    from transformer_head_scaled_sdpa_gb300 import binding, build
    if rank == 0:
        build.build()
    mdist.barrier(dev)
    build.build()  # no-op once built; loads on every rank
    w = inputs.BY_NAME[args.workload]
    case = inputs.generate(w, seed=mdist.rank_seed(w.seed, rank))
    stream = torch.cuda.Stream(device=dev)
    pairs = visible_pairs(w, case["key_lens"])
    flops_alg = 4.0 * w.d_k * pairs                 # per launch, this rank
    flops_nominal = w.flops()                       # 4 B H Lq Lk d_k, halved if causal
    elem = 2 if w.dtype == torch.bfloat16 else 4
    bytes_alg = elem * w.B * w.H * w.d_k * (2 * w.Lq + 2 * w.Lk)

    kernel_ms, max_total_ms, clocks, launches_per_step, bytes_in = measure_forward(
        w, case, args, dev, stream, rank, args.steps, args.warmup)
    kernel_label = fwd_kernel_label(w)
    n_sets = 1 if bytes_in > L2_BYTES else -(-2 * L2_BYTES // bytes_in)
    total_flops = mdist.sum_over_ranks(flops_nominal * args.steps, dev)
    total_flops_alg = mdist.sum_over_ranks(flops_alg * args.steps, dev)

    # end to end: pinned host buffers through the C ABI's host entry
    e2e = None
    if rank == 0 or world > 1:
        hq, hk, hv = (case[n].pin_memory() for n in ("q", "k", "v"))
        hout = torch.empty_like(hq).pin_memory()
        hlens = case["key_lens"].pin_memory() if case["key_lens"] is not None else None
        ws = torch.empty(binding.host_workspace_bytes(w.B, w.H, w.Lq, w.Lk, w.d_k, elem),
                         dtype=torch.uint8, device=dev)
        n_e2e = max(3, min(args.steps, 10))
        for _ in range(2):
            binding.mha_fwd_host(hq, hk, hv, hout, ws, mask_kind=w.mask_kind, key_lens=hlens,
                                 stream=stream)
        mdist.barrier(dev)
        torch.cuda.synchronize(dev)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n_e2e):
            binding.mha_fwd_host(hq, hk, hv, hout, ws, mask_kind=w.mask_kind, key_lens=hlens,
                                 stream=stream)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        e2e_ms = mdist.max_over_ranks(e0.elapsed_time(e1) / n_e2e, dev)
        e2e_flops = mdist.sum_over_ranks(flops_nominal, dev)
        h2d = bytes_in + (hlens.numel() * 4 if hlens is not None else 0)
        e2e = {"value": e2e_flops / (e2e_ms * 1e-3) / 1e12, "unit": UNIT,
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(hout.numel() * elem),
               "steps": n_e2e, "ms_per_step": e2e_ms,
               "path": "mha_fwd_host (C ABI): pinned host q,k,v -> device, kernel, out -> host"}
        del ws
        if rank == 0:
            link = host_link(dev, stream)
            e2e["host_link"] = link
            moved = (h2d + hout.numel() * elem) / (e2e_ms * 1e-3) / 1e9
            e2e["host_gbs"] = moved
            e2e["frac_host_link_both"] = moved / link["both_gbs"]

    if rank != 0:
        mdist.finish()
        return
    peaks, peak_src = load_peaks()
    value = total_flops / (max_total_ms * 1e-3) / 1e12
    achieved = flops_alg / (kernel_ms * 1e-3) / 1e12
    peak = float(peaks["bf16_tflops"])
    traffic = traffic_record(kernel_fingerprint("fwd_bf16_kernel"), w.name)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": max_total_ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if w.dtype == torch.bfloat16 else "f32",
        "data": "synthetic (seeded N(0,1) inputs, no dataset)",
        "config": workload_config(w, {
            "parallelism": f"replicas x{world} (no collective)",
            "inputs_exceed_l2": bytes_in * n_sets > L2_BYTES, "l2_flush": False,
            "input_sets_rotated": n_sets,
            "flops": "value: nominal 4*B*H*Lq*Lk*d_k (halved under the causal mask); "
                     "roofline: the (query, visible key) pairs",
            "flops_nominal_per_step_per_gpu": flops_nominal,
            "flops_algorithmic_per_step_per_gpu": flops_alg,
            **timing_config(args)}),
        "value_algorithmic": total_flops_alg / (max_total_ms * 1e-3) / 1e12,
        "pct_of_peak": 100.0 * value / world / peak,
        "pct_of_sustained_peak": 100.0 * value / world / float(
            peaks.get("bf16_tflops_sustained", peak)),
        "roofline": ({"bound": "tensor", "achieved": achieved, "peak": peak, "unit": UNIT,
                      "frac": achieved / peak, "traffic": traffic,
                      "peak_source": f"{peak_src} dense bf16 (burst)",
                      "kernel": kernel_label,
                      "kernel_ms": kernel_ms, "algorithmic_bytes": bytes_alg,
                      "achieved_gbs": bytes_alg / (kernel_ms * 1e-3) / 1e9}
                     if w.dtype == torch.bfloat16 else
                     # the float32 kernel runs on the CUDA cores: 152 SMs x 128
                     # FMA lanes x 2 flops x 2070 MHz (nominal)
                     {"bound": "alu", "achieved": achieved, "peak": F32_ALU_TFLOPS, "unit": UNIT,
                      "frac": achieved / F32_ALU_TFLOPS, "traffic": None,
                      "peak_source": "nominal fp32 FMA rate (152 x 128 x 2 x 2.07 GHz)",
                      "kernel": "fwd_f32_kernel", "kernel_ms": kernel_ms,
                      "algorithmic_bytes": bytes_alg,
                      "achieved_gbs": bytes_alg / (kernel_ms * 1e-3) / 1e9}),
        "clocks": clocks,
        "e2e": e2e,
        "gpu_launches": int(launches_per_step * args.steps),
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, case)
    if world == 1 and not args.no_sweep:
        # every configuration, each timed the same way (graph of >= 50 steps)
        rows = []
        sweep_steps = max(args.steps, 50)
        for name in SWEEP:
            wc = inputs.BY_NAME[name]
            if name == w.name:
                rows.append(config_record(wc, case, kernel_ms, launches_per_step, peaks,
                                          not args.no_cpu_baseline, kernel_label))
                continue
            c = inputs.generate(wc)
            k_ms, _, _, launches, _ = measure_forward(wc, c, args, dev, stream, rank,
                                                      sweep_steps, args.warmup)
            rows.append(config_record(wc, c, k_ms, launches, peaks, not args.no_cpu_baseline,
                                      fwd_kernel_label(wc)))
            del c
        line["configs"] = rows
    print(json.dumps(line), flush=True)
    mdist.finish()


# ---------------------------------------------------------------------------
# reference arm: the float64 oracle on the host cores
# ---------------------------------------------------------------------------
def run_reference(args):
    rank, world, _ = mdist.env_rank_world()
    if rank != 0:
        return
    import oracle
    w = inputs.BY_NAME[args.workload]
    case = inputs.generate(w)
    cores = oracle.default_threads()
    heads = [(b, h) for b in range(w.B) for h in range(w.H)]
    one = inputs.Workload(w.name, 1, 1, w.d_k, w.Lq, w.Lk, w.mask_kind, w.dtype)

    def run_heads(n, start):
        pairs = 0.0
        for i in range(n):
            b, h = heads[(start + i) % len(heads)]
            sub = {x: case[x][b:b + 1, :, h:h + 1] for x in ("q", "k", "v")}
            lens = case["key_lens"][b:b + 1] if case["key_lens"] is not None else None
            oracle.mha(sub["q"], sub["k"], sub["v"], w.mask_kind,
                       key_lens=lens.numpy() if lens is not None else None)
            pairs += visible_pairs(one, lens)
        return 4.0 * w.d_k * pairs

    t0 = time.perf_counter()
    run_heads(1, 0)
    t_head = time.perf_counter() - t0
    budget = 150.0 / max(1, args.steps + args.warmup)   # whole run within a few minutes
    per_step = max(1, int(budget / max(t_head, 1e-6)))
    for i in range(args.warmup):
        run_heads(per_step, i * per_step)
    t0 = time.perf_counter()
    flops = 0.0
    for i in range(args.steps):
        flops += run_heads(per_step, (args.warmup + i) * per_step)
    dt = time.perf_counter() - t0
    value = flops / dt / 1e12
    sample = (f"{per_step} whole (b, h) head(s) of {w.name} per step ({w.Lq}x{w.Lk}, d_k {w.d_k}, "
              f"{inputs.MASK_NAMES[w.mask_kind]}), float64 oracle, {cores} threads")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) inputs, no dataset)",
        "config": workload_config(w, {"parallelism": "host cores (OpenMP)"}),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


# ---------------------------------------------------------------------------
# decode steps
# ---------------------------------------------------------------------------
DEC_METRIC = "attention decode step GB/s (bf16 K/V cache read, 1 GB300) and % of measured HBM bandwidth"
DEC_UNIT = "GB/s"


def decode_bytes(w, lens):
    """Algorithmic bytes of one step: q and out once, the visible K and V rows."""
    visible = float(lens.clamp(0, w.Lk).to(torch.int64).sum().item())
    return 2.0 * visible * w.H * w.d_k * 2 + 2.0 * w.B * w.H * w.d_k * 2


def decode_config(w, extra=None):
    cfg = {"workload": w.name, "B": w.B, "sources": w.sources, "beams": w.beams, "H": w.H,
           "d_k": w.d_k, "Lk_capacity": w.Lk, "cache_len_range": [w.len_lo, w.len_hi],
           "input_scale": w.input_scale, "seed": w.seed,
           "layout": "q [B, H, d_k]; caches [B, Lk, H, d_k]"}
    if extra:
        cfg.update(extra)
    return cfg


def decode_oracle_rows(w, case, rows, start):
    """The oracle on `rows` (b, h) decode rows; returns the algorithmic bytes done."""
    import oracle
    done = 0.0
    for i in range(rows):
        r = (start + i) % (w.B * w.H)
        b, h = divmod(r, w.H)
        n = int(case["cache_lens"][b])
        q = case["q"][b:b + 1, h:h + 1].reshape(1, 1, 1, w.d_k)
        k = case["k_cache"][b:b + 1, :, h:h + 1]
        v = case["v_cache"][b:b + 1, :, h:h + 1]
        oracle.mha(q, k, v, inputs.MASK_KEY_PADDING,
                   key_lens=case["cache_lens"][b:b + 1].numpy())
        done += 2.0 * min(max(n, 0), w.Lk) * w.d_k * 2 + 2.0 * w.d_k * 2
    return done


def run_decode(args):
    rank, world = mdist.init("nccl")
    _, _, local_rank = mdist.env_rank_world()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    from transformer_head_scaled_sdpa_gb300 import binding, build
    if rank == 0:
        build.build()
    mdist.barrier(dev)
    build.build()
    w = inputs.DECODE_BY_NAME[args.workload]
    case = inputs.generate_decode(w, seed=mdist.rank_seed(w.seed, rank))
    g = {n: t.to(dev) for n, t in case.items()}
    bytes_alg = decode_bytes(w, case["cache_lens"])
    cache_bytes = 2 * g["k_cache"].numel() * 2
    n_sets = 1 if cache_bytes > L2_BYTES else -(-2 * L2_BYTES // cache_bytes)
    sets = [g] + [{n: t.clone() for n, t in g.items()} for _ in range(n_sets - 1)]
    outs = [torch.empty_like(g["q"]) for _ in range(n_sets)]
    ws = torch.empty(max(1, binding.decode_workspace_bytes(w.B, w.H, w.Lk, w.d_k)),
                     dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)
    cur = [0]

    def step():
        i = cur[0] % n_sets
        cur[0] += 1
        c = sets[i]
        binding.mha_decode(c["q"], c["k_cache"], c["v_cache"], c["cache_lens"], out=outs[i],
                           workspace=ws, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    rc = binding.mha_sync_status(stream)
    if rc != 0:
        raise binding.MhaError(rc, "warm-up")
    launches_per_step = binding.last_launch_info()["kernels"]
    step_ms, max_total_ms, clocks = timed_steps(step, args, dev, stream, rank, warm=False)
    rc = binding.mha_sync_status(stream)
    if rc != 0:
        raise binding.MhaError(rc, "timed region")
    total_bytes = mdist.sum_over_ranks(bytes_alg * args.steps, dev)

    # end to end through the public API: each step brings q (and the cache
    # lengths) from pinned host memory, runs the step on the resident cache and
    # reads the output back
    hq = case["q"].pin_memory()
    hlens = case["cache_lens"].pin_memory()
    hout = torch.empty_like(hq).pin_memory()
    dq = torch.empty_like(g["q"])
    dlens = torch.empty_like(g["cache_lens"])
    n_e2e = max(3, min(args.steps, 50))

    def e2e_step():
        dq.copy_(hq, non_blocking=True)
        dlens.copy_(hlens, non_blocking=True)
        binding.mha_decode(dq, g["k_cache"], g["v_cache"], dlens, out=outs[0], workspace=ws,
                           stream=stream)
        hout.copy_(outs[0], non_blocking=True)

    with torch.cuda.stream(stream):
        for _ in range(2):
            e2e_step()
    mdist.barrier(dev)
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(n_e2e):
            e2e_step()
        e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = mdist.max_over_ranks(e0.elapsed_time(e1) / n_e2e, dev)
    e2e_bytes = mdist.sum_over_ranks(bytes_alg, dev)
    if rank != 0:
        mdist.finish()
        return
    peaks, peak_src = load_peaks()
    peak = float(peaks["hbm_gbs"])
    value = total_bytes / (max_total_ms * 1e-3) / 1e9
    achieved = bytes_alg / (step_ms * 1e-3) / 1e9
    line = {
        "metric": DEC_METRIC, "value": value, "unit": DEC_UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": max_total_ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic (seeded N(0,1) inputs, no dataset)",
        "config": decode_config(w, {
            "parallelism": f"replicas x{world} (no collective)",
            "inputs_exceed_l2": cache_bytes * n_sets > L2_BYTES, "l2_flush": False,
            "input_sets_rotated": n_sets, "bytes_per_step_per_gpu": bytes_alg,
            "splits": binding.last_launch_info()["kernels"] > 1, **timing_config(args)}),
        "pct_of_peak": 100.0 * value / world / peak,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": DEC_UNIT,
                     "frac": achieved / peak,
                     "traffic": traffic_record(kernel_fingerprint("decode_split_kernel"), w.name, "decode_split_kernel"),
                     "peak_source": f"{peak_src} HBM copy bandwidth",
                     "kernel": "decode_split_kernel (+ decode_combine_kernel when split)",
                     "kernel_ms": step_ms, "algorithmic_bytes": bytes_alg},
        "clocks": clocks,
        "e2e": {"value": e2e_bytes / (e2e_ms * 1e-3) / 1e9, "unit": DEC_UNIT,
                "h2d_bytes_per_step": int(hq.numel() * 2 + hlens.numel() * 4),
                "d2h_bytes_per_step": int(hout.numel() * 2), "steps": n_e2e,
                "ms_per_step": e2e_ms,
                "path": "pinned host q, cache_lens -> device, mha_decode on the resident cache, "
                        "out -> host"},
        "gpu_launches": int(launches_per_step * args.steps),
    }
    if world == 1 and not args.no_cpu_baseline:
        import oracle
        t0 = time.perf_counter()
        done, rows = 0.0, 0
        while time.perf_counter() - t0 < 10.0 and rows < 4 * w.B * w.H:
            done += decode_oracle_rows(w, case, 8, rows)
            rows += 8
        dt = time.perf_counter() - t0
        line["cpu_baseline"] = {
            "value": done / dt / 1e9, "unit": DEC_UNIT, "cores": oracle.default_threads(),
            "kind": "oracle", "seconds": dt,
            "sample": f"{rows} (b, h) decode rows of {w.name} in float64, {dt:.1f} s wall"}
    print(json.dumps(line), flush=True)
    mdist.finish()


def run_reference_decode(args):
    rank, world, _ = mdist.env_rank_world()
    if rank != 0:
        return
    import oracle
    w = inputs.DECODE_BY_NAME[args.workload]
    case = inputs.generate_decode(w)
    cores = oracle.default_threads()
    t0 = time.perf_counter()
    decode_oracle_rows(w, case, 1, 0)
    t_row = time.perf_counter() - t0
    budget = 150.0 / max(1, args.steps + args.warmup)
    per_step = max(1, int(budget / max(t_row, 1e-6)))
    for i in range(args.warmup):
        decode_oracle_rows(w, case, per_step, i * per_step)
    t0 = time.perf_counter()
    done = 0.0
    for i in range(args.steps):
        done += decode_oracle_rows(w, case, per_step, (args.warmup + i) * per_step)
    dt = time.perf_counter() - t0
    value = done / dt / 1e9
    sample = f"{per_step} (b, h) decode row(s) of {w.name} per step, float64 oracle, {cores} threads"
    print(json.dumps({
        "impl": "reference", "metric": DEC_METRIC, "value": value, "unit": DEC_UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt * 1e3 / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded N(0,1) inputs, no dataset)",
        "config": decode_config(w, {"parallelism": "host cores (OpenMP)"}),
        "cpu_baseline": {"value": value, "unit": DEC_UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": DEC_UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


# ---------------------------------------------------------------------------
# backward pass
# ---------------------------------------------------------------------------
BWD_METRIC = "attention bwd TFLOP/s (bf16, 1 GB300; 2.5x forward flops) and % of dense BF16 tensor peak"


# ---------------------------------------------------------------------------
# the multi-head layer (projections around the attention)
# ---------------------------------------------------------------------------
LAYER_METRIC = ("multi-head attention layer TFLOP/s (bf16 Q/K/V and W^O projections on the "
                "library's tcgen05 GEMM + the attention kernel, 1 GB300) and % of measured dense "
                "bf16 peak")


def layer_sample(w, case, rows):
    """An exact sub-problem of the layer for the CPU oracle: sequence 0, and
    under the causal mask only its first ``rows`` query rows (they depend on
    x rows 0 .. rows-1 alone); otherwise the whole sequence."""
    n = min(rows, w.Lq) if (w.mask_kind & inputs.MASK_CAUSAL and not w.cross) else w.Lq
    sub = {"x": case["x"][:1, :n], "w_qkv": case["w_qkv"], "w_o": case["w_o"],
           "mem": case["mem"][:1] if case["mem"] is not None else None,
           "key_lens": case["key_lens"][:1] if case["key_lens"] is not None else None}
    one = inputs.LayerWorkload(w.name, 1, n, n if not w.cross else w.Lk, w.d_model, w.H, w.d_k,
                               w.mask_kind, cross=w.cross)
    return sub, one


def layer_oracle_baseline(w, case, budget_s=10.0):
    """The float64 layer oracle on growing exact samples within a budget."""
    import oracle
    rows = 64
    best = None
    t_all = time.perf_counter()
    while True:
        sub, one = layer_sample(w, case, rows)
        lens = sub["key_lens"].numpy() if sub["key_lens"] is not None else None
        t0 = time.perf_counter()
        oracle.mha_layer(sub["x"], sub["w_qkv"], sub["w_o"], w.H, mem=sub["mem"],
                         mask_kind=w.mask_kind, key_lens=lens)
        dt = time.perf_counter() - t0
        best = (one.flops(sub["key_lens"]) / dt / 1e12, dt, one.Lq)
        if one.Lq >= w.Lq or time.perf_counter() - t_all + 4 * dt > budget_s:
            break
        rows *= 2
    value, dt, n = best
    return {"value": value, "unit": UNIT, "cores": oracle.default_threads(), "kind": "oracle",
            "seconds": dt, "rows": n,
            "sample": f"sequence 0 of {w.name}, query rows 0..{n - 1} (an exact sub-problem: "
                      f"{'causal prefix' if w.mask_kind & inputs.MASK_CAUSAL else 'whole sequence'}), "
                      f"float64 numpy projections + the C attention oracle, {dt:.1f} s wall"}


def run_layer(args):
    rank, world = mdist.init("nccl")
    _, _, local_rank = mdist.env_rank_world()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    from transformer_head_scaled_sdpa_gb300 import binding, build
    if rank == 0:
        build.build()
    mdist.barrier(dev)
    build.build()
    w = inputs.LAYER_BY_NAME[args.workload]
    case = inputs.generate_layer(w, seed=mdist.rank_seed(w.seed, rank))
    g = {n: (t.to(dev) if t is not None else None) for n, t in case.items()}
    flops_alg = w.flops(case["key_lens"])
    y = torch.empty_like(g["x"])
    ws = torch.empty(max(1, binding.layer_workspace_bytes(w.B, w.Lq, w.Lk, w.d_model, w.H, w.d_k)),
                     dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)
    in_bytes = sum(t.numel() * 2 for n, t in g.items() if t is not None and n != "key_lens")

    def step():
        binding.mha_layer_fwd(g["x"], g["w_qkv"], g["w_o"], w.H, mem=g["mem"], mask_kind=w.mask_kind,
                              key_lens=g["key_lens"], y=y, workspace=ws, stream=stream)

    step_ms, max_total_ms, clocks = timed_steps(step, args, dev, stream, rank)
    rc = binding.mha_sync_status(stream)
    if rc != 0:
        raise binding.MhaError(rc, "timed region")
    launches_per_step = binding.last_launch_info()["kernels"]
    total_flops = mdist.sum_over_ranks(flops_alg * args.steps, dev)
    # end to end: x (and mem) from pinned host memory, y back; weights resident
    hx = case["x"].pin_memory()
    hm = case["mem"].pin_memory() if case["mem"] is not None else None
    hy = torch.empty_like(hx).pin_memory()
    dx = torch.empty_like(g["x"])
    dm = torch.empty_like(g["mem"]) if g["mem"] is not None else None
    n_e2e = max(3, min(args.steps, 20))

    def e2e_step():
        dx.copy_(hx, non_blocking=True)
        if dm is not None:
            dm.copy_(hm, non_blocking=True)
        binding.mha_layer_fwd(dx, g["w_qkv"], g["w_o"], w.H, mem=dm, mask_kind=w.mask_kind,
                              key_lens=g["key_lens"], y=y, workspace=ws, stream=stream)
        hy.copy_(y, non_blocking=True)

    with torch.cuda.stream(stream):
        e2e_step()
    mdist.barrier(dev)
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(n_e2e):
            e2e_step()
        e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = mdist.max_over_ranks(e0.elapsed_time(e1) / n_e2e, dev)
    e2e_flops = mdist.sum_over_ranks(flops_alg, dev)
    if rank != 0:
        mdist.finish()
        return
    peaks, peak_src = load_peaks()
    peak = float(peaks["bf16_tflops"])
    value = total_flops / (max_total_ms * 1e-3) / 1e12
    achieved = flops_alg / (step_ms * 1e-3) / 1e12
    cfg = {"workload": w.name, "B": w.B, "Lq": w.Lq, "Lk": w.Lk, "d_model": w.d_model, "H": w.H,
           "d_k": w.d_k, "mask": inputs.MASK_NAMES[w.mask_kind], "cross": w.cross,
           "seed": w.seed, "weights": "random (Xavier-scaled N(0, 1/fan_in), bf16)",
           "parallelism": f"replicas x{world} (no collective)",
           "inputs_exceed_l2": in_bytes > L2_BYTES, "l2_flush": False,
           "flops_per_step_per_gpu": flops_alg, **timing_config(args)}
    line = {
        "metric": LAYER_METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": max_total_ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) x, random weights, no dataset or trained model)",
        "config": cfg,
        "pct_of_peak": 100.0 * value / world / peak,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": UNIT,
                     "frac": achieved / peak, "traffic": None,
                     "peak_source": f"{peak_src} dense bf16 (burst)",
                     "kernel": "gemm_bf16_kernel projections + fwd_bf16_kernel (whole step)",
                     "kernel_ms": step_ms},
        "clocks": clocks,
        "e2e": {"value": e2e_flops / (e2e_ms * 1e-3) / 1e12, "unit": UNIT,
                "h2d_bytes_per_step": int(hx.numel() * 2 + (hm.numel() * 2 if hm is not None else 0)),
                "d2h_bytes_per_step": int(hy.numel() * 2), "steps": n_e2e, "ms_per_step": e2e_ms,
                "path": "pinned host x (and mem) -> device, mha_layer_fwd with resident weights, "
                        "y -> host"},
        # this library's own kernels: the projection GEMMs and the attention
        "gpu_launches": int(launches_per_step * args.steps),
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = layer_oracle_baseline(w, case)
    print(json.dumps(line), flush=True)
    mdist.finish()


def run_reference_layer(args):
    rank, world, _ = mdist.env_rank_world()
    if rank != 0:
        return
    w = inputs.LAYER_BY_NAME[args.workload]
    case = inputs.generate_layer(w)
    base = layer_oracle_baseline(w, case, budget_s=min(30.0, 120.0 / max(1, args.steps)))
    import oracle
    sub, one = layer_sample(w, case, base["rows"])
    lens = sub["key_lens"].numpy() if sub["key_lens"] is not None else None
    for _ in range(min(args.warmup, 3)):
        oracle.mha_layer(sub["x"], sub["w_qkv"], sub["w_o"], w.H, mem=sub["mem"],
                         mask_kind=w.mask_kind, key_lens=lens)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.mha_layer(sub["x"], sub["w_qkv"], sub["w_o"], w.H, mem=sub["mem"],
                         mask_kind=w.mask_kind, key_lens=lens)
    dt = time.perf_counter() - t0
    value = one.flops(sub["key_lens"]) * args.steps / dt / 1e12
    print(json.dumps({
        "impl": "reference", "metric": LAYER_METRIC, "value": value, "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt * 1e3 / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded, random weights)",
        "config": {"workload": w.name, "B": w.B, "Lq": w.Lq, "Lk": w.Lk, "d_model": w.d_model,
                   "H": w.H, "d_k": w.d_k, "mask": inputs.MASK_NAMES[w.mask_kind],
                   "parallelism": "host cores"},
        "cpu_baseline": dict(base, value=value),
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def run_bwd(args):
    rank, world = mdist.init("nccl")
    _, _, local_rank = mdist.env_rank_world()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    from transformer_head_scaled_sdpa_gb300 import binding, build
    if rank == 0:
        build.build()
    mdist.barrier(dev)
    build.build()
    w = inputs.BY_NAME[args.workload]
    if w.dtype != torch.bfloat16:
        raise SystemExit("--pass bwd needs a bf16 workload")
    seed = mdist.rank_seed(w.seed, rank)
    case = inputs.generate(w, seed=seed)
    dout_h = inputs.generate(w, seed=seed + 77)["q"]
    q, k, v = (case[n].to(dev) for n in ("q", "k", "v"))
    dout = dout_h.to(dev)
    lens = case["key_lens"].to(dev) if case["key_lens"] is not None else None
    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        out, lse = binding.mha_fwd(q, k, v, mask_kind=w.mask_kind, key_lens=lens,
                                   return_lse=True, stream=stream)
    dq, dk, dv = (torch.empty_like(t) for t in (q, k, v))
    ws = torch.empty(max(1, binding.lib().mha_bwd_workspace_bytes(w.B, w.H, w.Lq, w.Lk, w.d_k)),
                     dtype=torch.uint8, device=dev)
    flops_alg = 2.5 * 4.0 * w.d_k * visible_pairs(w, case["key_lens"])
    io = [q, k, v, out, dout, lse, dq, dk, dv]
    bytes_alg = sum(t.numel() * t.element_size() for t in io)

    def step():
        binding.mha_bwd(q, k, v, out, dout, lse, mask_kind=w.mask_kind, key_lens=lens, dq=dq,
                        dk=dk, dv=dv, workspace=ws, stream=stream)

    step_ms, max_total_ms, clocks = timed_steps(step, args, dev, stream, rank)
    rc = binding.mha_sync_status(stream)
    if rc != 0:
        raise binding.MhaError(rc, "timed region")
    launches_per_step = binding.last_launch_info()["kernels"]
    total_flops = mdist.sum_over_ranks(flops_alg * args.steps, dev)
    # end to end: host inputs (pinned) in, gradients out, every step
    host_in = [t.cpu().pin_memory() for t in (q, k, v, out, dout, lse)]
    host_out = [torch.empty_like(t, device="cpu").pin_memory() for t in (dq, dk, dv)]
    dev_in = [torch.empty_like(t) for t in (q, k, v, out, dout, lse)]
    n_e2e = max(3, min(args.steps, 10))

    def e2e_step():
        for d_, h_ in zip(dev_in, host_in):
            d_.copy_(h_, non_blocking=True)
        binding.mha_bwd(*dev_in, mask_kind=w.mask_kind, key_lens=lens, dq=dq, dk=dk, dv=dv,
                        workspace=ws, stream=stream)
        for h_, d_ in zip(host_out, (dq, dk, dv)):
            h_.copy_(d_, non_blocking=True)

    with torch.cuda.stream(stream):
        e2e_step()
    mdist.barrier(dev)
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(n_e2e):
            e2e_step()
        e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = mdist.max_over_ranks(e0.elapsed_time(e1) / n_e2e, dev)
    e2e_flops = mdist.sum_over_ranks(flops_alg, dev)
    if rank != 0:
        mdist.finish()
        return
    peaks, peak_src = load_peaks()
    peak = float(peaks["bf16_tflops"])
    value = total_flops / (max_total_ms * 1e-3) / 1e12
    achieved = flops_alg / (step_ms * 1e-3) / 1e12
    line = {
        "metric": BWD_METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": max_total_ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) inputs and dout, no dataset)",
        "config": workload_config(w, {"pass": "bwd", "parallelism": f"replicas x{world} (no collective)",
                                      "inputs_exceed_l2": bytes_alg > L2_BYTES, "l2_flush": False,
                                      "flops_per_step_per_gpu": flops_alg,
                                      **timing_config(args)}),
        "pct_of_peak": 100.0 * value / world / peak,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": UNIT,
                     "frac": achieved / peak, "traffic": None,
                     "peak_source": f"{peak_src} dense bf16 (burst)",
                     "kernel": "bwd_dq_kernel + bwd_dkdv_kernel (whole step)",
                     "kernel_ms": step_ms, "algorithmic_bytes": bytes_alg},
        "clocks": clocks,
        "e2e": {"value": e2e_flops / (e2e_ms * 1e-3) / 1e12, "unit": UNIT,
                "h2d_bytes_per_step": int(sum(t.numel() * t.element_size() for t in host_in)),
                "d2h_bytes_per_step": int(sum(t.numel() * t.element_size() for t in host_out)),
                "steps": n_e2e, "ms_per_step": e2e_ms,
                "path": "pinned host q,k,v,out,dout,lse -> device, mha_bwd, dq,dk,dv -> host"},
        "gpu_launches": int(launches_per_step * args.steps),
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = bwd_oracle_baseline(w, case, dout_h, 10.0)
    print(json.dumps(line), flush=True)
    mdist.finish()


def bwd_oracle_baseline(w, case, dout, budget_s):
    """The oracle's gradient on whole (b, h) heads within a time budget."""
    import oracle
    t0 = time.perf_counter()
    flops, heads = 0.0, 0
    one = inputs.Workload(w.name, 1, 1, w.d_k, w.Lq, w.Lk, w.mask_kind, w.dtype)
    while heads < w.B * w.H and (heads == 0 or time.perf_counter() - t0 < budget_s):
        b, h = divmod(heads, w.H)
        sub = {n: case[n][b:b + 1, :, h:h + 1] for n in ("q", "k", "v")}
        lens = case["key_lens"][b:b + 1] if case["key_lens"] is not None else None
        oracle.mha_bwd(sub["q"], sub["k"], sub["v"], dout[b:b + 1, :, h:h + 1], w.mask_kind,
                       key_lens=lens.numpy() if lens is not None else None)
        flops += 2.5 * 4.0 * w.d_k * visible_pairs(one, lens)
        heads += 1
    dt = time.perf_counter() - t0
    return {"value": flops / dt / 1e12, "unit": UNIT, "cores": oracle.default_threads(),
            "kind": "oracle", "seconds": dt,
            "sample": f"gradient of {heads} whole (b, h) head(s) of {w.name} in float64 "
                      f"(parallel over heads only), {dt:.1f} s wall"}


def run_reference_bwd(args):
    rank, world, _ = mdist.env_rank_world()
    if rank != 0:
        return
    import oracle
    w = inputs.BY_NAME[args.workload]
    case = inputs.generate(w)
    dout = inputs.generate(w, seed=w.seed + 77)["q"]
    budget = max(1.0, 150.0 / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        bwd_oracle_baseline(w, case, dout, budget)
    vals = [bwd_oracle_baseline(w, case, dout, budget) for _ in range(args.steps)]
    value = sum(x["value"] for x in vals) / len(vals)
    base = vals[-1]
    print(json.dumps({
        "impl": "reference", "metric": BWD_METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * sum(x["seconds"] for x in vals) / len(vals),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) inputs and dout, no dataset)",
        "config": workload_config(w, {"pass": "bwd", "parallelism": "host cores (OpenMP)"}),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": base["cores"], "kind": "oracle",
                         "sample": base["sample"]},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


# ---------------------------------------------------------------------------
# the projection GEMM alone (mha_gemm_bf16) against torch.matmul
# ---------------------------------------------------------------------------
GEMM_METRIC = "projection GEMM TFLOP/s (bf16, float32 accumulation, 1 GB300)"
# (M, N, K) of the layers' projections: GPT-3-like Q|K|V and W^O (B 4 x L 2048
# rows), a square reference, the base model's Q|K|V and W^O (32 x 128 rows)
GEMM_SHAPES = [(8192, 36864, 12288), (8192, 12288, 12288), (8192, 8192, 8192),
               (4096, 1536, 512), (4096, 512, 512)]


def run_gemm(args):
    rank, world = mdist.init("nccl")
    _, _, local_rank = mdist.env_rank_world()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    from transformer_head_scaled_sdpa_gb300 import binding, build
    if rank == 0:
        build.build()
    mdist.barrier(dev)
    build.build()
    peaks, peak_src = load_peaks()
    peak = float(peaks["bf16_tflops"])
    rows = []
    g = torch.Generator(device="cpu").manual_seed(4321)
    for M, N, K in GEMM_SHAPES:
        a = torch.randn(M, K, generator=g).to(torch.bfloat16).to(dev)
        b = (torch.randn(K, N, generator=g) / K ** 0.5).to(torch.bfloat16).to(dev)
        c = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
        flops = 2.0 * M * N * K
        res = {}
        for name, fn in (("ours", lambda: binding.mha_gemm_bf16(a, b, c)),
                         ("torch", lambda: torch.matmul(a, b, out=c))):
            for _ in range(args.warmup):
                fn()
            torch.cuda.synchronize(dev)
            n = max(3, int(2e12 / flops))
            best = float("inf")
            for _ in range(3):
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record()
                for _ in range(n):
                    fn()
                e1.record()
                torch.cuda.synchronize(dev)
                best = min(best, e0.elapsed_time(e1) / n)
            res[name] = flops / (best * 1e-3) / 1e12
        rc = binding.mha_sync_status()
        if rc != 0:
            raise binding.MhaError(rc, "gemm")
        rows.append({"M": M, "N": N, "K": K, "tflops": res["ours"], "torch_tflops": res["torch"],
                     "ratio_to_torch": res["ours"] / res["torch"], "frac": res["ours"] / peak})
        del a, b, c
    if rank == 0:
        first = rows[0]
        print(json.dumps({
            "metric": GEMM_METRIC, "value": first["tflops"], "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) x, N(0,1/K) weights)",
            "config": {"workload": "projection GEMMs", "shapes": GEMM_SHAPES,
                       "timing": "CUDA events around back-to-back calls, best of 3"},
            "roofline": {"bound": "tensor", "achieved": first["tflops"], "peak": peak,
                         "unit": UNIT, "frac": first["frac"], "traffic": None,
                         "peak_source": f"{peak_src} dense bf16 (burst)",
                         "kernel": "gemm_bf16_kernel"},
            "gemms": rows}), flush=True)
    mdist.finish()


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    # default: ~0.8 s timed on gpt3_causal, long enough for several clock samples
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="gpt3_causal",
                    choices=sorted(inputs.BY_NAME) + sorted(inputs.DECODE_BY_NAME) +
                    sorted(inputs.LAYER_BY_NAME))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--pass", dest="pass_", default="fwd", choices=["fwd", "bwd", "gemm"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sweep", action="store_true",
                    help="skip the per-configuration sweep of the default forward run")
    ap.add_argument("--eager", action="store_true",
                    help="issue the timed steps one by one instead of replaying a CUDA graph")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.steps < 1:
        ap.error("--steps must be >= 1")
    decode = args.workload in inputs.DECODE_BY_NAME
    if args.pass_ == "gemm":
        if args.impl == "reference":
            ap.error("--pass gemm has no reference arm")
        run_gemm(args)
        return
    if args.workload in inputs.LAYER_BY_NAME:
        if args.pass_ == "bwd":
            ap.error("--pass bwd applies to the attention workloads")
        (run_reference_layer if args.impl == "reference" else run_layer)(args)
        return
    if args.pass_ == "bwd":
        if decode:
            ap.error("--pass bwd applies to the forward workloads")
        (run_reference_bwd if args.impl == "reference" else run_bwd)(args)
    elif args.impl == "reference":
        (run_reference_decode if decode else run_reference)(args)
    else:
        (run_decode if decode else run_ours)(args)


if __name__ == "__main__":
    main()
