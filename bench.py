"""Throughput benchmark of the layerwise row-band VAE decode on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--no-cpu-baseline]

One step = one full decode (every op of the hot path) of the workload's seeded
latent with seeded random-init weights.  The default workload is the Z-Image
AutoencoderKL decoder at 1024x1024 (latent 1x16x128x128, bf16, 8 row bands).
Prints ONE JSON line on rank 0.

--impl ours       the CUDA library through its C ABI (device-resident inputs for
                  `value`; host buffers with the copies inside the timed region for
                  `e2e`), plus roofline, clocks and the CPU oracle baseline.
--impl reference  the float64 CPU oracle, timed on the host cores on a bounded
                  sample of the workload (a latent crop), in the same metric.

Multi-GPU (torchrun): every rank decodes its own replica (the decode is not split
across GPUs here); value = all ranks' pixels / max-over-ranks time.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "VAE decode Mpixel/s at 1024² bf16 on 1 GB300; conv tensor-pipe util %"
UNIT = "Mpixel/s"
# Pages' dense single-GPU Z-Image BF16 1024x1024 decode: 105.97 ms on one RTX PRO 6000
# Blackwell Server Edition with pretrained weights, i.e. 1048576 px / 105.97 ms.
PAGES_DENSE_MPIXS = 1048576 / 105.97e-3 / 1e6
L2_FLUSH_BYTES = 256 << 20
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def out_pixels(w: synth.Workload) -> int:
    shp = w.latent_shape
    f = 2 ** sum(1 for u in w.arch.stage_upsample if u)
    if w.arch.family == "kl2d":
        f *= w.arch.latent_patch          # a patched latent is unpatchified to twice the grid first
        return shp[0] * shp[2] * f * shp[3] * f
    t = shp[2]
    for u in w.arch.stage_upsample:
        if u == 2:
            t = 2 * t - 1
    return shp[0] * t * shp[3] * f * shp[4] * f


# The dominant kernel of the step (largest share of the ncu launch list) and the
# committed summary of its measured DRAM traffic.  The traffic figure is used only
# while the kernel source still hashes to the value recorded with the counters.
DOMINANT_KERNEL = "conv_halo_t"
DOMINANT_SOURCE = os.path.join(ROOT, "row_band_layerwise_gb300", "csrc", "conv_halo_t.cu")
TRAFFIC_SUMMARY = os.path.join(ROOT, "profiles", "conv_halo_t_kernel_kl_zimage_1024_traffic.md")


def measured_traffic(workload: str):
    """(DRAM bytes per launch, note) from the committed ncu summary, or (None, why)."""
    import hashlib
    import re
    if workload != "kl_zimage_1024":
        return None, "no ncu traffic summary for this workload"
    try:
        text = open(TRAFFIC_SUMMARY).read()
    except OSError:
        return None, "no ncu traffic summary committed"
    m_hash = re.search(r"source_sha256:\s*([0-9a-f]{64})", text)
    m_bytes = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not (m_hash and m_bytes):
        return None, "ncu traffic summary unreadable"
    cur = hashlib.sha256(open(DOMINANT_SOURCE, "rb").read()).hexdigest()
    if cur != m_hash.group(1):
        return None, "kernel changed since the ncu counters were taken"
    return float(m_bytes.group(1)), os.path.relpath(TRAFFIC_SUMMARY, ROOT)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured (MEASURED_PEAKS.json)"
    return dict(FALLBACK_PEAKS), "fallback (no MEASURED_PEAKS.json)"


def max_over_ranks(value: float, device=None) -> float:
    """The largest `value` over all ranks of the default process group (itself when there is
    none).  Works on any backend: the tensor lives on `device` (CUDA for NCCL, CPU for gloo)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device or "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(world_size: int, steps: int, pixels_per_step: int, seconds: float) -> float:
    """Whole-job Mpixel/s of `world_size` replicas that each decoded `steps` steps, timed by the
    slowest rank (weak scaling: every rank decodes the full workload)."""
    return world_size * steps * pixels_per_step / seconds / 1e6


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


# ---------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"vaedec_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                    power.append(float(parts[3]))
                except ValueError:
                    continue
                for nm, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(nm)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(power) if power else None}


# ---------------------------------------------------------------- CPU oracle
def oracle_sample(w: synth.Workload, max_rows: int, max_cols: int):
    """A crop of the workload's seeded latent (same weights, same decoder)."""
    z = synth.make_latent(w.latent_shape, w.dtype)
    if w.arch.family == "kl2d":
        zc = z[:1, :, :max_rows, :max_cols]
    else:
        zc = z[:1, :, :, :max_rows, :max_cols]
    return np.ascontiguousarray(zc)


def time_oracle(w: synth.Workload, W, zc, repeats: int = 1):
    from oracle import decoder as odec
    times = []
    for _ in range(repeats):
        t0 = time.perf_counter()
        y = odec.decode(w.arch, W, zc)
        times.append(time.perf_counter() - t0)
    px = int(np.prod(y.shape)) // y.shape[1]
    return px, times


def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def sample_shape(w, small: bool = False):
    """Latent crop (rows, cols) timed on the CPU: about 10-30 s of float64 work on a
    16-core host for the baseline, a few seconds per step for the reference arm."""
    if w.arch.family == "kl2d":
        return (16, 16) if small else (64, 64)
    return (4, 8) if small else (16, 16)


def run_reference(args, w: synth.Workload):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    W = synth.make_weights(w.arch, w.dtype)
    rows, cols = sample_shape(w, small=True)
    zc = oracle_sample(w, rows, cols)
    px = None
    for _ in range(args.warmup):
        px, _ = time_oracle(w, W, zc)
    times = []
    for _ in range(args.steps):
        px, t = time_oracle(w, W, zc)
        times += t
    total = sum(times)
    value = args.steps * px / total / 1e6
    cores = cpu_cores()
    sample = (f"latent crop {tuple(zc.shape)} of the seeded workload latent ({px} output pixels per step), "
              f"same weights; float64 numpy oracle")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded latent crop, random-init weights)",
        "config": {"workload": w.name, "description": w.description, "sample": sample},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- ours
def run_ours(args, w: synth.Workload):
    import torch
    import row_band_layerwise_gb300 as rbl

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)

    W = synth.make_weights(w.arch, w.dtype)
    z = synth.make_latent(w.latent_shape, w.dtype)
    shp = w.latent_shape
    max_latent = (shp[0], 1, shp[2], shp[3]) if len(shp) == 4 else (shp[0], shp[2], shp[3], shp[4])
    dec = rbl.Decoder(w.arch, W, w.dtype, max_latent)
    tdt = dec.torch_dtype
    zd = torch.from_numpy(z).to(dev).to(tdt).contiguous()
    out = torch.empty(dec.output_shape(shp), dtype=tdt, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    nb = args.bands or w.n_bands

    def barrier():
        if ws > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(dev)

    axis = rbl.band_axis(shp, nb, args.band_axis)
    torch.cuda.synchronize(dev)
    torch.cuda.reset_peak_memory_stats(dev)
    alloc0 = torch.cuda.memory_allocated(dev)
    for _ in range(args.warmup):
        dec.decode(zd, nb, out=out, axis=axis)
    dec.sync()
    torch_delta = torch.cuda.max_memory_allocated(dev) - alloc0   # allocations made by the decodes

    # op list (for the per-kernel-kind roofline)
    ops = dec.ops(shp, nb)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    launches0 = dec.launch_count()
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    barrier()
    for i in range(args.steps):
        flush.zero_()                       # evict L2 between steps (outside the step events)
        starts[i].record(stream)
        dec.decode(zd, nb, out=out, stream=stream, axis=axis)
        ends[i].record(stream)
    barrier()
    clock_info = clocks.stop()
    launches = dec.launch_count() - launches0
    dec.sync()
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    # per-op CUDA-event times from one more decode, outside the timed steps (an event between every
    # two ops changes how consecutive kernels overlap, so the timed steps run without them)
    dec.profile(True)
    flush.zero_()
    dec.decode(zd, nb, out=out, stream=stream, axis=axis)
    dec.sync()
    per_op = dec.profile_read()
    dec.profile(False)
    total_ms = max_over_ranks(sum(step_ms), dev)
    px = out_pixels(w)
    value = replica_throughput(ws, args.steps, px, total_ms / 1e3)

    # roofline of the dominant kernel: its conv ops' algorithmic flops over their event-timed durations
    conv_ms = sum(ms for d, ms in zip(ops, per_op) if d["kind"] == "conv")
    dom = [(d, ms) for d, ms in zip(ops, per_op) if d["kind"] == "conv" and d.get("kernel") == DOMINANT_KERNEL]
    dom_ms = sum(ms for _, ms in dom)
    dom_flops = sum(float(d["flops"]) for d, _ in dom)
    # multiply-adds the tensor cores execute: less than the algorithmic count where an upsample conv
    # runs in its exact two-by-two phase form (7 weight taps per phase instead of 9)
    dom_exec = sum(float(d.get("exec_flops", d["flops"])) for d, _ in dom)
    traffic, traffic_src = measured_traffic(w.name)
    attn_ms = sum(ms for d, ms in zip(ops, per_op) if d["kind"] == "attention")
    attn_flops = sum(float(d["flops"]) for d in ops if d["kind"] == "attention")
    norm_ms = sum(ms for d, ms in zip(ops, per_op) if d["kind"] in ("groupnorm", "rmsnorm"))
    all_flops = sum(float(d.get("flops", 0.0)) for d in ops if d["kind"] in ("conv", "attention"))
    peaks, peak_src = load_peaks()
    # burst peak: the decode runs at the maximum SM clock for ~10 ms per step, not in the
    # seconds-long power-capped loop the sustained figure was measured in
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    achieved = dom_flops / (dom_ms / 1e3) / 1e12 if dom_ms > 0 else 0.0

    # end to end through the C ABI with host buffers (copies inside the timed region)
    zh = torch.from_numpy(z).to(tdt).pin_memory()
    oh = torch.empty(dec.output_shape(shp), dtype=tdt).pin_memory()
    for _ in range(max(1, args.warmup // 2)):
        dec.decode_host(zh, oh, nb)
    barrier()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        dec.decode_host(zh, oh, nb)
    e2e_s = max_over_ranks(time.perf_counter() - t0, dev)
    e2e_value = replica_throughput(ws, args.steps, px, e2e_s)

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        rows, cols = sample_shape(w)
        zc = oracle_sample(w, rows, cols)
        cpx, ct = time_oracle(w, W, zc)
        cpu = {"value": cpx / ct[0] / 1e6, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
               "sample": f"one float64 oracle decode of a latent crop {tuple(zc.shape)} of the workload "
                         f"({cpx} output pixels, {ct[0]:.1f} s, numpy BLAS on all cores)"}

    if rank == 0:
        line = {
            "impl": "ours", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": total_ms / args.steps,
            "median_ms_per_step": statistics.median(step_ms), "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": value / PAGES_DENSE_MPIXS if w.name == "kl_zimage_1024" else None,
            "dtype": "bf16" if w.dtype == "bf16" else "f32",
            "data": "synthetic (seeded N(0,1) latent, seeded fan-in uniform weights)",
            "config": {"workload": w.name, "description": w.description, "n_bands": nb, "band_axis": axis,
                       "latent": list(shp), "output_pixels_per_step": px,
                       "l2": f"{L2_FLUSH_BYTES >> 20} MiB buffer written between steps, outside the step events",
                       "parallelism": "replicas" if ws > 1 else "single GPU",
                       "per_op_times": "CUDA events per op on the decode stream, one decode after the timed "
                                       "steps (the timed steps record no per-op events)",
                       "workspace_bytes": dec.workspace_bytes(),
                       "memory": {"workspace_bytes": dec.workspace_bytes(),
                                  "output_bytes": out.numel() * out.element_size(),
                                  "torch_peak_delta_bytes": int(torch_delta),
                                  "peak_extra_bytes": dec.workspace_bytes() + out.numel() * out.element_size()
                                  + int(torch_delta),
                                  "note": "device memory beyond weights and latent: the handle's workspace "
                                          "(allocated once at create), the caller's output, and any allocation "
                                          "during the decodes (max_memory_allocated delta)"},
                       "vs_baseline_ref": "pages' dense single-GPU Z-Image BF16 1024x1024 decode, 105.97 ms on "
                                          "RTX PRO 6000 Blackwell (context only)"},
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                         "frac": achieved / peak if peak else None, "traffic": traffic,
                         "kernel": f"{DOMINANT_KERNEL}_kernel", "launches_per_step": len(dom),
                         "flops_per_step": dom_flops, "kernel_ms_per_step": dom_ms,
                         "executed_flops_per_step": dom_exec,
                         "executed_tflops": dom_exec / (dom_ms / 1e3) / 1e12 if dom_ms > 0 else None,
                         "executed_frac": dom_exec / (dom_ms / 1e3) / 1e12 / peak if dom_ms > 0 and peak else None,
                         "conv_tensor_util_pct": 100.0 * achieved / peak if peak else None,
                         "conv_tensor_util_note": "the metric's conv tensor-pipe utilisation: the dominant conv "
                                                  "kernel's algorithmic flops per second over the measured bf16 "
                                                  "peak; ncu's sm__pipe_tensor_cycles_active for sampled launches "
                                                  "is in profiles/conv_halo_t_kernel_kl_zimage_512_full.md",
                         "per_launch": "algorithmic flops (nearest-2x then 3x3 counted as 3x3 on the high-resolution "
                                       "output) / CUDA-event duration, summed over its launches; executed_* count "
                                       "the multiply-adds the tensor cores run",
                         "traffic_source": traffic_src,
                         "peak_source": f"bf16_tflops (burst), {peak_src}",
                         "sm_mhz_median": clock_info.get("sm_mhz"),
                         "decode_frac": (all_flops / (statistics.median(step_ms) / 1e3) / 1e12 / peak
                                         if peak else None),
                         "decode_flops_per_step": all_flops,
                         "decode_frac_note": "algorithmic conv + attention flops of one decode / median step "
                                             "time / peak"},
            "breakdown_ms": {"conv": conv_ms, "attention": attn_ms, "norm": norm_ms,
                             "other": sum(per_op) - conv_ms - attn_ms - norm_ms,
                             "attention_tflops": attn_flops / (attn_ms / 1e3) / 1e12 if attn_ms else None},
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": zh.numel() * zh.element_size(),
                    "d2h_bytes_per_step": oh.numel() * oh.element_size()},
            "gpu_launches": launches,
            "clocks": clock_info,
        }
        print(json.dumps(line), flush=True)
    dec.close()
    if ws > 1:
        torch.distributed.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="kl_zimage_1024", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--bands", type=int, default=0, help="override the workload's band count")
    ap.add_argument("--band-axis", default="height", choices=["height", "width", "auto"],
                    help="band split axis of the device-timed decodes (e2e always uses height bands)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    w = synth.WORKLOADS[args.workload]
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
