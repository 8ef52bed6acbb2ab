"""Throughput of the FLUX-class VAE decoder on GB300: decode Mpix/s.

One step = one full decode (de-normalise, conv_in, mid block, up blocks,
norm_out, conv_out) of a seeded synthetic latent with random-init weights, the
whole chain running in this repository's sm_103a kernels.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload decoder_1024]
  python bench.py --impl reference ...   # the float64 CPU oracle on host cores

Multi-GPU (torchrun): every rank decodes its own latent (independent images,
no exchange between ranks: "replicas", weak scaling); the timed region is
bracketed by barriers and the max time over ranks is used.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import vae_synth as S  # noqa: E402

WORKLOADS = {
    "decoder_1024": dict(latent=(1, 16, 128, 128), seed=S.seed_of("decoder_1024"),
                         text="FLUX-class AutoencoderKL decoder, latent [1,16,128,128] -> RGB "
                              "[1,3,1024,1024], random init"),
    "decoder_256": dict(latent=(1, 16, 32, 32), seed=S.seed_of("decoder_256"),
                        text="FLUX-class AutoencoderKL decoder, latent [1,16,32,32] -> RGB "
                             "[1,3,256,256], random init"),
    "decoder_512": dict(latent=(1, 16, 64, 64), seed=S.seed_of("decoder_512_b4"),
                        text="FLUX-class AutoencoderKL decoder, latent [1,16,64,64] -> RGB "
                             "[1,3,512,512], random init (profiling size)"),
    "decoder_512_b4": dict(latent=(4, 16, 64, 64), seed=S.seed_of("decoder_512_b4"),
                           text="FLUX-class AutoencoderKL decoder, latent [4,16,64,64] -> RGB "
                                "[4,3,512,512], random init"),
}
METRIC = "VAE decode Mpix/s"
# Nominal dense tensor rates (PFLOP/s): TF32 1.1 vs BF16 2.25 (context only: the
# roofline fraction is taken against the TF32 MMA rate measured in the run).
TF32_OVER_BF16 = 1.1 / 2.25
FALLBACK_PEAKS = dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0)


def out_pixels(latent):
    n, _, h, w = latent
    return n * 8 * h * 8 * w


# ---------------------------------------------------------------- distributed helpers
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def rank_seed(seed, rank):
    """Each rank decodes a different latent (independent images)."""
    return seed + 7919 * rank


def reduce_max(value, dist=None):
    """Max of a float over all ranks (identity without a process group)."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(value)
    import torch
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(value)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(dist=None):
    if dist is not None and dist.is_initialized() and dist.get_world_size() > 1:
        dist.barrier()


# ---------------------------------------------------------------- peaks / clocks
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.gpu_index)], stdout=self.f,
                stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (FileNotFoundError, OSError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        with open(self.path) as f:
            for ln in f:
                parts = [p.strip() for p in ln.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(v):
            try:
                return float(v)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        pw = [num(r[3]) for r in rows if num(r[3]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4)
                          if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(pw) if pw else None,
                "samples": len(rows), "reasons": reasons}


def igemm_source_sha():
    import hashlib
    src = b"".join(open(os.path.join(ROOT, "diffusion_vae_decoder_gb300", "csrc", f), "rb").read()
                   for f in ("igemm.cu", "igemm_kernel.cuh"))
    return hashlib.sha256(src).hexdigest()


def conv_traffic_ratio(path=None):
    """DRAM bytes over algorithmic bytes of the implicit-GEMM conv, from the
    committed machine-readable ncu summary (profiles/igemm_traffic.json:
    single launches at single-op sweep shapes) -- (None, None) when the
    summary is missing or was taken on other kernel source (the kernel has
    changed since the counters were read)."""
    path = path or os.path.join(ROOT, "profiles", "igemm_traffic.json")
    if not os.path.exists(path):
        return None, None
    with open(path) as f:
        data = json.load(f)
    if data.get("igemm_sha256") != igemm_source_sha():
        return None, None
    return float(data["dram_over_algorithmic"]), data


# ---------------------------------------------------------------- CPU oracle timing
def time_oracle_decode(latent, seed, repeats=1):
    """Float64 CPU oracle decode of one latent; returns (seconds per decode, Mpix)."""
    import oracle
    w = S.make_decoder_weights("flux", seed)
    z = S.make_latent(latent, seed)
    t0 = time.perf_counter()
    for _ in range(repeats):
        oracle.decode(z, w, S.SCALING_FACTOR, S.SHIFT_FACTOR, 4)
    dt = (time.perf_counter() - t0) / repeats
    return dt, out_pixels(latent) / 1e6


def measure_tf32_peak(pkg, seconds=0.3):
    """TF32 tensor-pipe rate of this GPU (TFLOP/s) from the library's MMA-loop
    microkernel, with the SM clock sampled while it runs."""
    pkg.vae_measure_tf32_mma(2000)  # warm-up / calibration
    tf, ms, _ = pkg.vae_measure_tf32_mma(20000)
    iters = max(20000, int(20000 * seconds * 1e3 / max(ms, 1e-3)))
    return tf, iters


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# ---------------------------------------------------------------- reference arm
def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    wl = WORKLOADS[args.workload]
    sample = (1, 16, 16, 16)
    for _ in range(args.warmup):
        time_oracle_decode(sample, wl["seed"])
    total = 0.0
    for _ in range(args.steps):
        dt, mpix = time_oracle_decode(sample, wl["seed"])
        total += dt
    value = args.steps * mpix / total
    cores = host_cores()
    desc = ("float64 numpy oracle (per-tap BLAS matmuls) decoding latent [1,16,16,16] -> "
            "128x128 with the same architecture, one decode per step")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "Mpix/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, "text": wl["text"], "sample": desc},
        "cpu_baseline": {"value": value, "unit": "Mpix/s", "cores": cores, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": "Mpix/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- our arm
def run_ours(args):
    import torch

    import diffusion_vae_decoder_gb300 as pkg

    world, rank, local = dist_env()
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    wl = WORKLOADS[args.workload]
    latent = wl["latent"]
    seed = rank_seed(wl["seed"], rank)

    weights = S.make_decoder_weights("flux", wl["seed"])
    chain = pkg.VaeChain(weights, n_up_blocks=4)
    z_host = torch.from_numpy(S.make_latent(latent, seed)).pin_memory()
    z = z_host.to(dev)
    n, _, h, w = latent
    out = torch.empty((n, 3, 8 * h, 8 * w), dtype=torch.float32, device=dev)
    ws = torch.empty(chain.workspace_size(n, h, w), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    for _ in range(args.warmup):
        chain.decode(z, out=out, ws=ws)
    torch.cuda.synchronize()
    assert pkg.vae_device_error() == 0

    # ---- the decode captured once into a CUDA graph; the timed region
    # replays it. A second capture carries the step profiler's CUDA events
    # (two event-record nodes per step, which slow the decode by a few
    # percent); right after the timed region it is replayed over the same
    # number of steps, and its last replay gives the per-step durations that
    # the roofline is computed from.
    launches0 = pkg.vae_kernel_launch_count()
    graph = chain.capture_graph(z, out, ws)
    launches_per_decode = pkg.vae_kernel_launch_count() - launches0
    chain.profile(True)
    pgraph = chain.capture_graph(z, out, ws)
    chain.profile(False)
    graph.replay()
    pgraph.replay()
    torch.cuda.synchronize()
    gpu_index = local
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        ids = [v for v in vis.split(",") if v.strip()]
        if local < len(ids) and ids[local].strip().isdigit():
            gpu_index = int(ids[local])
    sampler = ClockSampler(gpu_index)
    with sampler:
        barrier(dist)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            graph.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        barrier(dist)
        p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        p0.record(stream)
        for _ in range(args.steps):
            pgraph.replay()
        p1.record(stream)
        torch.cuda.synchronize()
    launches = launches_per_decode * args.steps
    ms = e0.elapsed_time(e1) / args.steps
    ms_profiled = p0.elapsed_time(p1) / args.steps
    recs = chain.profile_read()  # the events of the last profiled replay
    if args.detail and rank == 0:
        for i, r in enumerate(recs):
            rate = (f"{r['flops'] / r['ms'] / 1e9:8.1f} TF/s" if r["flops"] else
                    f"{r['bytes'] / r['ms'] / 1e6:8.1f} GB/s")
            print(f"step {i:3d} {r['kind']:14s} kernels {r['kernels']:2d} {r['ms']:8.4f} ms {rate}",
                  file=sys.stderr)
    chain.profile(False)
    assert pkg.vae_device_error() == 0
    ms_max = reduce_max(ms, dist)
    mpix = out_pixels(latent) / 1e6
    value = world * mpix / (ms_max / 1e3)
    n_prof = 1  # one decode's worth of step records

    # ---- roofline of the dominant kernel (the implicit-GEMM conv) and of
    # GroupNorm. The conv's denominator is this GPU's TF32 tensor-pipe rate,
    # measured right here by the library's MMA-loop microkernel with the SM
    # clock sampled while it runs (the timed decode's clock is sampled above).
    peaks, peak_src = load_peaks()
    with ClockSampler(gpu_index) as psampler:
        _, iters = measure_tf32_peak(pkg)
        tf32_peak, tf32_ms, _ = pkg.vae_measure_tf32_mma(iters)
    tf32_clocks = psampler.summary()
    bf16_derived = peaks["bf16_tflops"] * TF32_OVER_BF16
    conv = [r for r in recs if r["kind"] in ("conv3x3", "upsample_conv")]
    gn = [r for r in recs if r["kind"] == "groupnorm"]
    conv_ms = sum(r["ms"] for r in conv)  # per decode
    conv_tflops = sum(r["flops"] for r in conv) / (conv_ms / 1e3) / 1e12
    gn_ms = sum(r["ms"] for r in gn)
    gn_gbs = sum(r["bytes"] for r in gn) / (gn_ms / 1e3) / 1e9
    head = [r for r in recs if r["kind"] == "head"]
    head_ms = sum(r["ms"] for r in head)
    head_gbs = sum(r["bytes"] for r in head) / (head_ms / 1e3) / 1e9 if head_ms > 0 else None
    step_ms_sum = sum(r["ms"] for r in recs) / n_prof
    by_kind = {}
    for r in recs:
        k = by_kind.setdefault(r["kind"], dict(ms=0.0, flops=0.0, bytes=0.0, steps=0))
        k["ms"] += r["ms"] / n_prof
        k["flops"] += r["flops"] / n_prof
        k["bytes"] += r["bytes"] / n_prof
        k["steps"] += 1
    for k in by_kind.values():
        k["steps"] //= n_prof

    # ---- end to end through the public API, host buffers, copies inside:
    # every step copies its latent from pinned host memory, runs the captured
    # decode and reads its RGB back into pinned host memory. Two buffer sets
    # let step i's read-back (on a copy stream) overlap step i+1's decode, as
    # a serving loop would pipeline them.
    h2d = z_host.numel() * 4
    zs = [z, torch.empty_like(z)]
    outs = [out, torch.empty_like(out)]
    graphs = [chain.capture_graph(zs[b], outs[b], ws) for b in range(2)]
    out_hosts = [torch.empty(out.shape, dtype=torch.float32).pin_memory() for _ in range(2)]
    d2h = out_hosts[0].numel() * 4
    copy_stream = torch.cuda.Stream()
    decoded = [torch.cuda.Event() for _ in range(2)]
    for b in range(2):  # warm both graphs
        graphs[b].replay()
    torch.cuda.synchronize()
    barrier(dist)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    read_back = [None, None]
    for i in range(args.steps):
        b = i & 1
        if read_back[b] is not None:  # outs[b] is free once its read-back is done
            stream.wait_event(read_back[b])
        zs[b].copy_(z_host, non_blocking=True)
        graphs[b].replay()
        decoded[b].record(stream)
        copy_stream.wait_event(decoded[b])
        with torch.cuda.stream(copy_stream):
            out_hosts[b].copy_(outs[b], non_blocking=True)
            read_back[b] = torch.cuda.Event()
            read_back[b].record(copy_stream)
    torch.cuda.synchronize()
    e2e_ms = reduce_max((time.perf_counter() - t0) * 1e3 / args.steps, dist)
    assert pkg.vae_device_error() == 0
    barrier(dist)
    e2e_value = world * mpix / (e2e_ms / 1e3)

    # DRAM traffic per conv launch: the decode's algorithmic bytes per conv
    # launch (input, output, residual, shortcut input once) times the
    # DRAM/algorithmic ratio ncu measured on single launches of this kernel.
    ratio, traffic_src = conv_traffic_ratio()
    conv_launches = sum(r["kernels"] for r in conv)
    alg_per_launch = sum(r["bytes"] for r in conv) / max(conv_launches, 1)
    traffic = alg_per_launch * ratio if ratio else None
    traffic_entry = None
    if traffic_src:
        traffic_entry = {"dram_over_algorithmic": ratio,
                         "algorithmic_bytes_per_launch": alg_per_launch,
                         "conv_launches_per_decode": conv_launches,
                         "captures": [c["shape"] for c in traffic_src["captures"]]}
    extras = None
    if rank == 0 and world == 1 and not args.no_extras:
        extras = run_extras(pkg, tf32_peak, gpu_index)
    line = None
    if rank == 0:
        cpu = None
        if not args.no_cpu_baseline and world == 1:
            sample = (1, 16, 32, 32)
            dt, smpix = time_oracle_decode(sample, wl["seed"])
            cpu = {"value": smpix / dt, "unit": "Mpix/s", "cores": host_cores(), "kind": "oracle",
                   "sample": "float64 numpy oracle decoding one latent [1,16,32,32] -> 256x256 "
                             f"with the same architecture ({dt:.1f} s)"}
        line = {
            "metric": METRIC, "value": value, "unit": "Mpix/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "tf32",
            "data": "synthetic",
            "config": {"workload": args.workload, "text": wl["text"],
                       "latent": list(latent), "global_batch": latent[0] * world,
                       "parallelism": f"replicas{world}",
                       "l2": "no flush: every step streams several GB of activations, far "
                             "beyond the 129 MB L2"},
            "roofline": {"bound": "tensor", "kernel": "igemm_kernel (3x3 / upsample conv)",
                         "achieved": conv_tflops, "peak": tf32_peak, "unit": "TFLOP/s",
                         "frac": conv_tflops / tf32_peak,
                         "traffic": traffic,
                         "traffic_source": traffic_entry,
                         "peak_source": "measured in this run: tcgen05 kind::tf32 MMA loop on "
                                        "every SM, operands resident in shared memory "
                                        f"({tf32_ms:.0f} ms; SM clock median "
                                        f"{tf32_clocks.get('sm_mhz')} MHz)",
                         "frac_vs_bf16_burst_derived": conv_tflops / bf16_derived,
                         "bf16_burst_derived_peak": bf16_derived,
                         "share_of_step": conv_ms / n_prof / ms_profiled,
                         "measured": "CUDA events around every conv step inside the profiled "
                                     "capture of the decode, last of the K profiled replays run "
                                     "right after the timed region"},
            "roofline_groupnorm": {"bound": "hbm", "achieved": gn_gbs, "peak": peaks["hbm_gbs"],
                                   "unit": "GB/s", "frac": gn_gbs / peaks["hbm_gbs"],
                                   "bytes_per_element": "8 (read + write) where the statistics "
                                                        "come from the producing conv, 12 for "
                                                        "the two-pass GroupNorms"},
            "roofline_head": None if head_gbs is None else {
                "bound": "hbm", "achieved": head_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": head_gbs / peaks["hbm_gbs"],
                "bytes_per_pixel": "4 * C_in read + 4 * C_out written (norm_out + conv_out step, "
                                   "its GroupNorm finalize included)"},
            "steps_by_kind": by_kind, "profiled_ms_per_step": ms_profiled,
            "profiled_steps_sum_ms": step_ms_sum,
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": "Mpix/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                    "timed": "host clock around K steps of: pinned latent -> device, graph "
                             "replay, RGB -> pinned host on a copy stream (read-back of step i "
                             "overlaps the decode of step i+1; two buffer sets)"},
            "gpu_launches": int(launches),
            "launches_per_decode": int(launches_per_decode),
            "clocks": sampler.summary(),
            "extra_workloads": extras,
        }
        print(json.dumps(line), flush=True)
    chain.close()
    if dist is not None:
        dist.destroy_process_group()
    return 0


def _graph_decode_stats(pkg, arch, latent, seed, steps):
    """Device time per decode of one latent (CUDA-graph replays, CUDA events)
    and the conv steps' TFLOP/s from a profiled capture."""
    import torch
    chain = pkg.VaeChain(S.make_decoder_weights(arch, seed), n_up_blocks=4)
    n, _, h, w = latent
    z = torch.from_numpy(S.make_latent(latent, seed)).cuda()
    out = torch.empty((n, 3, 8 * h, 8 * w), device="cuda")
    ws = torch.empty(chain.workspace_size(n, h, w), dtype=torch.uint8, device="cuda")
    for _ in range(3):
        chain.decode(z, out=out, ws=ws)
    graph = chain.capture_graph(z, out, ws)
    chain.profile(True)
    pgraph = chain.capture_graph(z, out, ws)
    chain.profile(False)
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        graph.replay()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    pgraph.replay()
    torch.cuda.synchronize()
    recs = chain.profile_read()
    chain.close()
    assert pkg.vae_device_error() == 0
    conv = [r for r in recs if r["kind"] in ("conv3x3", "upsample_conv")]
    conv_ms = sum(r["ms"] for r in conv)
    return ms, sum(r["flops"] for r in conv) / (conv_ms / 1e3) / 1e12, conv_ms


def run_extras(pkg, tf32_peak, gpu_index):
    """The other configured workloads, each on its own (rank 0, one GPU):
    the 256^2 decode and the batch-4 512^2 decode (Mpix/s), the tiny decoder
    (latency), the 3-D causal conv stack [1,128,17,128,128] (conv TFLOP/s)."""
    import torch
    out = {}
    ms, conv_tf, conv_ms = _graph_decode_stats(pkg, "flux", (1, 16, 32, 32),
                                               S.seed_of("decoder_256"), 200)
    out["decoder_256"] = {"value": out_pixels((1, 16, 32, 32)) / 1e6 / (ms / 1e3),
                          "unit": "Mpix/s", "ms_per_step": ms, "steps": 200,
                          "conv_tflops": conv_tf, "conv_frac": conv_tf / tf32_peak,
                          "conv_ms_per_step": conv_ms}
    lat4 = WORKLOADS["decoder_512_b4"]["latent"]
    ms, conv_tf, conv_ms = _graph_decode_stats(pkg, "flux", lat4, WORKLOADS["decoder_512_b4"]["seed"],
                                               20)
    out["decoder_512_b4"] = {"value": out_pixels(lat4) / 1e6 / (ms / 1e3), "unit": "Mpix/s",
                             "ms_per_step": ms, "steps": 20, "conv_tflops": conv_tf,
                             "conv_frac": conv_tf / tf32_peak, "conv_ms_per_step": conv_ms}
    ms, conv_tf, _ = _graph_decode_stats(pkg, "tiny", (1, 16, 8, 8), S.seed_of("tiny_decoder"),
                                         500)
    out["tiny_decoder"] = {"latency_ms": ms, "value": out_pixels((1, 16, 8, 8)) / 1e6 / (ms / 1e3),
                           "unit": "Mpix/s", "steps": 500}
    # 3-D causal conv stack, NDHWC (the kernels' layout): five 3x3x3 convs with
    # GroupNorm+SiLU and the residual every two layers.
    shape = S.WORKLOADS["causal3d_stack"]["shape"]
    x, layers = S.make_causal_stack(shape, 5, S.seed_of("causal3d_stack"))
    xd = torch.from_numpy(np.ascontiguousarray(np.moveaxis(x, 1, -1))).cuda()
    dl = [{k: torch.from_numpy(v).cuda() for k, v in L.items()} for L in layers]
    y = torch.empty_like(xd)
    n, c, t, h, w = shape
    flops_conv = 2.0 * c * c * 27 * n * t * h * w
    for _ in range(3):
        pkg.vae_causal_stack(xd, dl, layout=pkg.VAE_NHWC, out=y)
    one = torch.empty_like(xd)
    for _ in range(3):
        pkg.vae_conv3d_causal(xd, dl[0]["weight"], dl[0]["bias"], layout=pkg.VAE_NHWC, out=one)
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    ev[0].record()
    for _ in range(5):
        pkg.vae_causal_stack(xd, dl, layout=pkg.VAE_NHWC, out=y)
    ev[1].record()
    ev[2].record()
    for _ in range(10):
        pkg.vae_conv3d_causal(xd, dl[0]["weight"], dl[0]["bias"], layout=pkg.VAE_NHWC, out=one)
    ev[3].record()
    torch.cuda.synchronize()
    assert pkg.vae_device_error() == 0
    stack_ms = ev[0].elapsed_time(ev[1]) / 5
    conv_ms = ev[2].elapsed_time(ev[3]) / 10
    out["causal3d_stack"] = {
        "shape": list(shape), "stack_ms": stack_ms,
        "stack_conv_tflops": 5 * flops_conv / (stack_ms / 1e3) / 1e12,
        "conv_ms": conv_ms, "conv_tflops": flops_conv / (conv_ms / 1e3) / 1e12,
        "conv_frac": flops_conv / (conv_ms / 1e3) / 1e12 / tf32_peak,
        "note": "stack = five convs + five GroupNorm+SiLU (+ weight packing), NDHWC; conv = one "
                "vae_conv3d_causal call (its weight packing included)"}
    return out


SWEEP = [(128, 512), (256, 256), (512, 128), (512, 64)]  # (channels, input side)


def time_op(op, c, hw, steps, warmup):
    """One op of the single-op sweep (batch 1, NHWC, the chain's internal layout;
    inputs N(0,1), weights N(0, 1/(Cin*9))), timed with CUDA events.

    Every timed iteration is preceded by a 256 MB write that evicts L2; the
    iterations are queued back to back (one synchronize at the end), so the
    host enqueues the op while the GPU is still busy with the flush and the
    events time the op's kernels, not the host's launch latency. (The write
    is followed by a 256 MB read, so the op does not pay for writing back
    the flush's dirty lines.) The convs
    run on weights packed once (vae_conv2d_pack / vae_upsample_conv_pack);
    the packing is timed on its own, the same way, as pack_ms."""
    import torch

    import diffusion_vae_decoder_gb300 as pkg

    x = torch.from_numpy(S.make_normal((1, hw, hw, c), 31)).cuda()
    wt, b = S.make_conv_params(c, c, 3, 32)
    wt, b = torch.from_numpy(wt).cuda(), torch.from_numpy(b).cuda()
    g, be = (torch.from_numpy(a).cuda() for a in S.make_norm_params(c, 33))
    pack_fn = None
    if op == "conv":
        out = torch.empty_like(x)
        pack_fn = lambda: pkg.vae_conv2d_pack(wt, b)  # noqa: E731
        pk = pack_fn()
        fn = lambda: pkg.vae_conv2d_packed(x, pk, layout=pkg.VAE_NHWC, out=out)  # noqa: E731
        work, unit = 2.0 * c * c * 9 * hw * hw, "TFLOP/s"
    elif op == "upsample_conv":
        out = torch.empty((1, 2 * hw, 2 * hw, c), device="cuda")
        pack_fn = lambda: pkg.vae_upsample_conv_pack(wt, b)  # noqa: E731
        pk = pack_fn()
        fn = lambda: pkg.vae_upsample_conv_packed(x, pk, layout=pkg.VAE_NHWC, out=out)  # noqa: E731
        # executed work: four parity 2x2 convs, 4 taps per output pixel
        work, unit = 2.0 * c * c * 4 * 4 * hw * hw, "TFLOP/s"
    else:
        out = torch.empty_like(x)
        fn = lambda: pkg.vae_groupnorm_silu(x, g, be, layout=pkg.VAE_NHWC, out=out)  # noqa: E731
        work, unit = 12.0 * c * hw * hw, "GB/s"
    # L2 eviction between timed iterations: write one 256 MB buffer, then
    # read another, so that L2 ends up holding clean lines of unrelated data
    # (a write alone would leave it full of dirty lines whose write-back
    # would land inside the next timed op)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    flush_r = torch.ones(64 << 20, dtype=torch.float32, device="cuda")

    def timed(f):
        for _ in range(warmup):
            f()
        torch.cuda.synchronize()
        events = []
        for _ in range(steps):
            flush.zero_()  # evict L2 between timed iterations
            flush_r.sum()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            f()
            e1.record()
            events.append((e0, e1))
        torch.cuda.synchronize()
        return [e0.elapsed_time(e1) for e0, e1 in events]

    times = timed(fn)
    pack_ms = statistics.median(timed(pack_fn)) if pack_fn else None
    assert pkg.vae_device_error() == 0
    ms = statistics.median(times)
    rate = work / (ms / 1e3) / (1e12 if unit == "TFLOP/s" else 1e9)
    peaks, src = load_peaks()
    peak = (peaks["bf16_tflops"] * TF32_OVER_BF16 if unit == "TFLOP/s" else peaks["hbm_gbs"])
    return {"op": op, "c": c, "hw": hw, "layout": "NHWC", "ms_median": ms,
            "ms_min": min(times), "pack_ms": pack_ms, "rate": rate, "unit": unit, "peak": peak,
            "frac": rate / peak, "peak_source": src + " burst",
            "l2": "flushed between iterations (256 MB write, then 256 MB read)"}


def run_op(args):
    """`--op conv|upsample_conv|groupnorm`: one op at --c / --hw; `--op sweep`:
    every op at every shape of the single-op sweep, one JSON line each."""
    import torch

    torch.cuda.set_device(0)
    if args.op == "sweep":
        for op in ("conv", "upsample_conv", "groupnorm"):
            for c, hw in SWEEP:
                print(json.dumps(time_op(op, c, hw, args.steps, args.warmup)), flush=True)
        return 0
    print(json.dumps(time_op(args.op, args.c, args.hw, args.steps, args.warmup)), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="decoder_1024")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the other workloads (256^2 decode, tiny decoder, 3-D stack)")
    ap.add_argument("--detail", action="store_true",
                    help="also print every profiled step of one decode (stderr)")
    ap.add_argument("--op", choices=["conv", "upsample_conv", "groupnorm", "sweep"], default=None,
                    help="time one op of the single-op sweep (or all of them: sweep) "
                         "instead of the decoder")
    ap.add_argument("--c", type=int, default=128)
    ap.add_argument("--hw", type=int, default=512)
    args = ap.parse_args(argv)
    args.warmup = max(args.warmup, 3)  # at least 3 untimed warm-up steps
    if args.op:
        return run_op(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
