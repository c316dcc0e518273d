#!/usr/bin/env python
"""Benchmark: bf16 decode of a 720p x 81-frame video latent through libvaedec on GB300.

Metric: decoded Mframe-px/s = B * 81 * 704 * 1280 / decode time / 1e6 (whole job, all ranks).
Default workload: the Wan-shaped decoder (latent [1, 48, 21, 44, 80] -> pixels [1, 3, 81, 704, 1280],
stage channels 1024/1024/512/256, mid attention), random-init weights, seeded synthetic latent.

One JSON line on rank 0 with the contract's keys plus:
  roofline      the dominant kernel (tcgen05 causal conv) inside the timed decodes: algorithmic
                FLOPs / CUDA-event time over all its launches, against the measured bf16 peak
  kernels       the same per kernel class (conv, group norm stats/apply, attention GEMMs, ...)
  ops           the op-level workloads: PatchGroupNorm+SiLU, channel RMS norm+SiLU, causal conv 512->512,
                tile blend
  extra         the LTX-shaped 720p x 81f decode (1x4 and 2x4 patches), the batch-2 overlap-tiled LTX
                decode (45 tiles -> [2,3,129,1088,1920]), the Wan-shaped decode with e4m3 conv operands and
                the LTX-shaped encode of 720p x 81f, the LTX-shaped decode in fp32 (3 x TF32 convs):
                Mframe-px/s, conv fraction, per-kernel table
  cpu_baseline  the CPU oracle on a bounded sample of the same decode (first 2 latent frames of one
                full-width latent row), host cores
N > 1 (torchrun): each rank decodes its own latent (independent videos, weak scaling), no
collective on the data path; barriers and the max over ranks bracket the timed region.
--impl reference times the CPU oracle (the reference arm) on rank 0.
--workload ltx / wan_rms: the LTX-shaped decoder, or the Wan-shaped one with channel RMS norms.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from patch_tiled_causal_gb300 import synth  # noqa: E402

FRAME_PX_720P_81 = 81 * 704 * 1280


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def _src_sha(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "patch_tiled_causal_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def _traffic(kernel):
    """DRAM bytes per launch from the committed ncu summary, if the kernel source is unchanged."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    if not os.path.exists(p):
        return None
    try:
        with open(p) as f:
            d = json.load(f)
        e = d.get(kernel)
        if e and e.get("src_sha") == _src_sha(e["src_files"]):
            return e
    except Exception:
        return None
    return None


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms while running."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index=0):
        self.proc = None
        self.path = os.path.join("/tmp", f"vae_clocks_{os.getpid()}.csv")
        self.gpu = gpu_index

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.fh,
                                         stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        sm, smax, pw, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                try:
                    pw.append(float(parts[3]))
                except ValueError:
                    pass
                for n, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w": statistics.median(pw) if pw else None}


# ------------------------------------------------------------------------------------- CPU oracle
_PARAMS = {}


def oracle_sample(cfg, crop_thw, seed=0):
    """Time the CPU oracle (Tier B, float32) decoding a crop (first frames, top latent rows, left
    latent columns) of the workload's latent; returns (decoded frame-px, seconds).  The parameters
    are drawn once per workload, outside the timing."""
    from oracle import decoder as odec
    b, c, t, h, w = cfg.latent_shape
    ct, ch, cw = crop_thw
    sub = dataclasses.replace(cfg, latent_shape=(b, c, ct, ch, cw))
    if cfg.name not in _PARAMS:
        _PARAMS[cfg.name] = synth.draw_params(cfg, seed)
    p = _PARAMS[cfg.name]
    z = synth.draw_latent(cfg, seed)[:, :, :ct, :ch, :cw].copy()
    t0 = time.perf_counter()
    y = odec.decode(sub, p, z, tier="B")
    dt = time.perf_counter() - t0
    frame_px = y.shape[0] * y.shape[2] * y.shape[3] * y.shape[4]
    return frame_px, dt


# The oracle's bounded sample: the first 2 latent frames (-> 5 output frames) of one full-width row of
# latent pixels, so every layer runs its real channel counts over a full image row (realistic BLAS
# shapes); ~15 s per sample on 16 host cores.  The reference arm times one such sample per step.
SAMPLE_ROWS = 1
SAMPLE_FRAMES = 2
METRIC = "decoded Mframe-px/s at 720p x 81f bf16"


def sample_crop(cfg):
    return (SAMPLE_FRAMES, SAMPLE_ROWS, cfg.latent_shape[4])


def _crop_text(cfg, crop):
    return (f"{cfg.name} decode of the first {crop[0]} latent frames x {crop[1]} full-width row(s) of {crop[2]} latent "
            f"pixels (of {cfg.latent_shape[2]} x {cfg.latent_shape[3]}x{cfg.latent_shape[4]}), Tier B float32 "
            f"(numpy BLAS)")


def run_reference(args, cfg):
    crop = sample_crop(cfg)
    for _ in range(args.warmup):
        oracle_sample(cfg, crop)
    times, fpx = [], 0
    for _ in range(args.steps):
        fpx, dt = oracle_sample(cfg, crop)
        times.append(dt)
    total = sum(times)
    v = fpx * args.steps / total / 1e6
    cores = os.cpu_count()
    line = {"impl": "reference", "metric": METRIC,
            "value": v, "unit": "Mframe-px/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1000 * total / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": f"{cfg.name}-shaped decoder, latent {list(cfg.latent_shape)} -> "
                                   f"{list(cfg.output_shape())}; each step the CPU oracle on a bounded sample",
                       "l2": "n/a (CPU)"},
            "cpu_baseline": {"value": v, "unit": "Mframe-px/s", "cores": cores, "kind": "oracle",
                             "sample": _crop_text(cfg, crop)},
            "e2e": {"value": v, "unit": "Mframe-px/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------------------------- multi-rank
def latent_seed(rank: int) -> int:
    """Each rank decodes its own video: the latent of rank r is drawn from seed r."""
    return rank


def max_over_ranks(seconds: float, dist=None, device="cpu") -> float:
    """The timed region's length is the slowest rank's (all_reduce MAX; identity on one rank)."""
    if dist is None:
        return seconds
    import torch
    t = torch.tensor([seconds], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def throughput(frame_px_per_rank: int, steps: int, world: int, seconds: float) -> float:
    """Whole-job Mframe-px/s: every rank decodes steps videos of frame_px_per_rank each."""
    return frame_px_per_rank * steps * world / seconds / 1e6


# ------------------------------------------------------------------------------------- GPU arm
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="wan", choices=["wan", "ltx", "wan_rms"],
                    help="wan_rms: the Wan-shaped decoder with channel RMS norms instead of group norms")
    ap.add_argument("--patches", default="1x4", help="patch grid h x w of the timed decode")
    ap.add_argument("--no-ops", action="store_true", help="skip the op-level workloads")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU-oracle baseline")
    ap.add_argument("--no-extra", action="store_true", help="skip the LTX-shaped and tiled decode sub-lines")
    ap.add_argument("--only", default="all", choices=["all", "decode", "ops", "encode"],
                    help="run only the decode or only the op workloads (profiling runs)")
    ap.add_argument("--latent-frames", type=int, default=0,
                    help="decode only the first N latent frames (0: all; small values for profiler captures)")
    ap.add_argument("--blend-small", action="store_true",
                    help="op-level blend of the tiled LTX plan on batch 1 and 9 latent frames (profiler captures)")
    ap.add_argument("--ops-frames", type=int, default=0,
                    help="frames of the pixel-head op workloads (0: 81; smaller values for profiler captures)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    cfg = {"wan": synth.WAN, "ltx": synth.LTX, "wan_rms": synth.WAN_RMS}[args.workload]
    if args.latent_frames:
        shp = cfg.latent_shape
        cfg = dataclasses.replace(cfg, latent_shape=(shp[0], shp[1], args.latent_frames, shp[3], shp[4]))

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            run_reference(args, cfg)
        return

    import torch
    from patch_tiled_causal_gb300 import build, vaedec

    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    build.build()
    vaedec.load()
    peaks = _peaks()
    stream = torch.cuda.current_stream()

    if args.only == "ops":
        flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
        print(json.dumps({"ops": run_ops(args, torch, vaedec, peaks, flush), "peaks": peaks}), flush=True)
        return
    if args.only == "encode":  # the LTX-shaped encode alone (profiling runs)
        flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
        print(json.dumps({"ltx_encode_1x4": run_ltx_encode(args, torch, vaedec, peaks, flush, stream)}), flush=True)
        return
    if args.only == "decode":
        args.no_ops = args.no_cpu = args.no_extra = True

    nph, npw = (int(v) for v in args.patches.lower().split("x"))
    params = synth.draw_params(cfg, 0)
    latent_np = synth.draw_latent(cfg, seed=latent_seed(rank))
    dec = vaedec.Decoder(cfg, params, vaedec.VAE_BF16)
    del params
    dec.reserve(cfg.latent_shape, nph, npw)
    latent = torch.from_numpy(latent_np).cuda()
    out = torch.empty(dec.output_shape(latent.shape), dtype=torch.bfloat16, device="cuda")
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")  # > L2 (129 MB)

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    for _ in range(args.warmup):
        dec.decode(latent, out, nph, npw)
    code, msg = vaedec.last_error(dec.h)
    if code:
        raise RuntimeError(f"decode failed: {msg}")

    # ---- timed region: device-resident inputs, L2 flushed between steps, events on the stream
    sampler = ClockSampler(local)
    sampler.start()
    dec.profile(True)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    barrier()
    for a, b in evs:
        flush.zero_()
        a.record(stream)
        dec.decode(latent, out, nph, npw)
        b.record(stream)
    barrier()
    clocks = sampler.stop()
    prof = dec.profile_read()
    dec.profile(False)
    step_ms = [a.elapsed_time(b) for a, b in evs]
    t_max = max_over_ranks(sum(step_ms) / 1000.0, dist, "cuda")
    code, msg = vaedec.last_error(dec.h)
    if code:
        raise RuntimeError(f"decode failed in the timed region: {msg}")
    frame_px = out.shape[0] * out.shape[2] * out.shape[3] * out.shape[4]
    value = throughput(frame_px, args.steps, world, t_max)
    launches = sum(v["launches"] for v in prof.values()) // args.steps

    # ---- end to end through the public API: pinned host latent in, pinned host pixels out.  The headline
    # path is vae_decode_host (temporal chunks, the copies of one chunk overlapping the decode of the
    # next on a second stream); the serial path (copy in, vae_decode, copy out) is reported beside it.
    h_lat = torch.from_numpy(latent_np).pin_memory()
    h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    d_lat = torch.empty_like(latent)

    def e2e_host():
        dec.decode_host(h_lat, h_out, nph, npw)

    def e2e_serial():
        d_lat.copy_(h_lat, non_blocking=True)
        dec.decode(d_lat, out, nph, npw)
        h_out.copy_(out, non_blocking=True)

    def e2e_time(fn):
        for _ in range(2):
            fn()
        eev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
        barrier()
        for a, b in eev:
            flush.zero_()
            a.record(stream)
            fn()
            b.record(stream)
        barrier()
        return throughput(frame_px, args.steps, world,
                          max_over_ranks(sum(a.elapsed_time(b) for a, b in eev) / 1000.0, dist, "cuda"))

    e2e_sampler = ClockSampler(local)
    e2e_sampler.start()
    e2e_value = e2e_time(e2e_host)
    e2e_clocks = e2e_sampler.stop()
    e2e_serial_value = e2e_time(e2e_serial)
    code, msg = vaedec.last_error(dec.h)
    if code:
        raise RuntimeError(f"end-to-end decode failed: {msg}")

    kernels = kernel_table(prof, args.steps, peaks)
    conv = conv_totals(prof)
    conv_tf = conv["flops"] / (conv["ms"] / 1e3) / 1e12
    tr = _traffic(f"conv_tc_decode_{cfg.name}")
    roofline = {"bound": "tensor", "kernel": "conv_tc (tcgen05 implicit-GEMM causal conv), all launches of the decode",
                "achieved": conv_tf, "peak": peaks["bf16_tflops_sustained"], "unit": "TFLOP/s",
                "frac": conv_tf / peaks["bf16_tflops_sustained"],
                "peak_kind": f"bf16 dense, sustained, {'of measured' if peaks['source'] == 'measured' else 'of fallback'}",
                "traffic": tr["bytes_per_launch"] if tr else None,
                "flops_per_launch": conv["flops"] / conv["launches"],
                "ms_per_launch": conv["ms"] / conv["launches"]}
    if tr:
        roofline["traffic_note"] = tr.get("note", "")

    ops = None
    if not args.no_ops and rank == 0:
        ops = run_ops(args, torch, vaedec, peaks, flush)
    extra = None
    if not args.no_extra and rank == 0 and args.workload == "wan":
        dec.close()  # frees the Wan decoder's workspace before the LTX decoders are built
        torch.cuda.empty_cache()
        extra = run_ltx(args, torch, vaedec, peaks, flush, stream)
        extra["wan_fp8_1x4"] = run_wan_fp8(args, torch, vaedec, peaks, flush, stream)
        extra["ltx_encode_1x4"] = run_ltx_encode(args, torch, vaedec, peaks, flush, stream)
        extra["ltx_fp32_1x4"] = run_ltx_fp32(args, torch, vaedec, peaks, flush, stream)

    cpu = None
    if not args.no_cpu and rank == 0 and world == 1:
        crop = sample_crop(cfg)
        fpx, dt = oracle_sample(cfg, crop)
        cpu = {"value": fpx / dt / 1e6, "unit": "Mframe-px/s", "cores": os.cpu_count(), "kind": "oracle",
               "sample": _crop_text(cfg, crop) + f", {fpx} frame-px in {dt:.1f} s"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "Mframe-px/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * t_max / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) latent, N(0,1/fan_in) random-init weights)",
            "config": {"workload": f"{cfg.name}-shaped causal VAE decoder, latent {list(cfg.latent_shape)} -> "
                                   f"pixels {list(out.shape)}, {nph}x{npw} spatial patches",
                       "global_batch": out.shape[0] * world, "frames": out.shape[2],
                       "resolution": f"{out.shape[3]}x{out.shape[4]}", "patches": f"{nph}x{npw}",
                       "parallelism": f"replicas x{world} (independent videos)", "l2": "flushed between steps"},
            "e2e": {"value": e2e_value, "unit": "Mframe-px/s", "h2d_bytes_per_step": latent.numel() * 4,
                    "d2h_bytes_per_step": out.numel() * out.element_size(),
                    "api": "vae_decode_host (pinned host latent in, pinned host pixels out; temporal chunks with "
                           "the copies overlapping the decode on a second stream)",
                    "serial_value": e2e_serial_value,
                    "clocks": {"sm_mhz": e2e_clocks["sm_mhz"], "power_w": e2e_clocks.get("power_w"),
                               "reasons": e2e_clocks["reasons"]}},
            "gpu_launches": launches,
            "roofline": roofline,
            "kernels": kernels,
            "clocks": clocks,
            "cpu_baseline": cpu,
            "ops": ops,
            "extra": extra,
            "peaks": peaks,
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


def kernel_table(prof, steps, peaks):
    """Per kernel class: launches and device time per step, share, and the fraction of its roofline."""
    kernels = {}
    total = max(sum(x["ms"] for x in prof.values()), 1e-9)
    for k, v in sorted(prof.items(), key=lambda kv: -kv[1]["ms"]):
        e = {"launches_per_step": v["launches"] // steps, "ms_per_step": v["ms"] / steps, "share": v["ms"] / total}
        if v["flops"]:
            e["tflops"] = v["flops"] / (v["ms"] / 1e3) / 1e12
            e["frac_of_bf16_sustained"] = e["tflops"] / peaks["bf16_tflops_sustained"]
        if v["bytes"]:
            e["gbs"] = v["bytes"] / (v["ms"] / 1e3) / 1e9
            e["frac_of_hbm"] = e["gbs"] / peaks["hbm_gbs"]
        kernels[k] = e
    return kernels


def conv_totals(prof):
    """The tcgen05 conv kernel over all its launches: the body convs plus the pixel head (conv_head)."""
    conv = {k: sum(prof.get(c, {}).get(k, 0) for c in ("conv_tc", "conv_head")) for k in ("flops", "ms", "launches")}
    return conv if conv["launches"] else {"flops": 0.0, "ms": 1.0, "launches": 1}


def timed_decodes(torch, dec, fn, steps, warmup, flush, stream):
    """Run fn (one decode) warmup times, then steps timed times with L2 flushed before each; returns
    (ms per decode from CUDA events on the launching stream, per-kernel profile of the timed decodes)."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    dec.profile(True)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for a, b in evs:
        flush.zero_()
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize()
    prof = dec.profile_read()
    dec.profile(False)
    return sum(a.elapsed_time(b) for a, b in evs) / steps, prof


def run_wan_fp8(args, torch, vd, peaks, flush, stream):
    """The Wan-shaped 720p x 81f decode (1x4 patches) with e4m3 conv operands (VAE_FP8)."""
    cfg = synth.WAN
    params = synth.draw_params(cfg, 0)
    dec = vd.Decoder(cfg, params, vd.VAE_FP8)
    del params
    z = torch.from_numpy(synth.draw_latent(cfg, 0)).cuda()
    out = torch.empty(dec.output_shape(z.shape), dtype=torch.bfloat16, device="cuda")
    ms, prof = timed_decodes(torch, dec, lambda: dec.decode(z, out, 1, 4), args.steps, args.warmup, flush, stream)
    code, msg = vd.last_error(dec.h)
    if code:
        raise RuntimeError(f"fp8 decode failed: {msg}")
    dec.close()
    fpx = out.shape[0] * out.shape[2] * out.shape[3] * out.shape[4]
    del z, out
    torch.cuda.empty_cache()
    return {"workload": f"wan-shaped decoder, latent {list(cfg.latent_shape)}, 1x4 patches, e4m3 operands for the "
                        "residual-block and up-sampler convs (conv_in, conv_out, attention bf16), pixels bf16",
            "value": fpx / ms / 1e3, "unit": "Mframe-px/s", "ms_per_step": ms, "dtype": "fp8 (e4m3) conv operands",
            "kernels": kernel_table(prof, args.steps, peaks)}


def run_ltx_fp32(args, torch, vd, peaks, flush, stream):
    """The LTX-shaped 720p x 81f decode (1x4 patches) in fp32 storage with the convs as three TF32
    products per fp32 product on the tensor cores (VAE_FP32_TC)."""
    cfg = synth.LTX
    params = synth.draw_params(cfg, 0)
    dec = vd.Decoder(cfg, params, vd.VAE_FP32_TC)
    del params
    z = torch.from_numpy(synth.draw_latent(cfg, 0)).cuda()
    out = torch.empty(dec.output_shape(z.shape), dtype=torch.float32, device="cuda")
    ms, prof = timed_decodes(torch, dec, lambda: dec.decode(z, out, 1, 4), args.steps, args.warmup, flush, stream)
    code, msg = vd.last_error(dec.h)
    if code:
        raise RuntimeError(f"fp32 decode failed: {msg}")
    dec.close()
    fpx = out.shape[0] * out.shape[2] * out.shape[3] * out.shape[4]
    conv = conv_totals(prof)
    tf = conv["flops"] / (conv["ms"] / 1e3) / 1e12
    # three TF32 products per fp32 product: the effective peak is a third of the tf32 dense peak, taken as
    # the measured sustained bf16 figure x the nominal tf32 / bf16 ratio (1.1 / 2.25)
    eff_peak = peaks["bf16_tflops_sustained"] * (1.1 / 2.25) / 3.0
    del z, out
    torch.cuda.empty_cache()
    return {"workload": f"ltx-shaped decoder, latent {list(cfg.latent_shape)}, 1x4 patches, fp32 storage, convs as "
                        "3 x TF32 products on the tensor cores, pixels fp32",
            "value": fpx / ms / 1e3, "unit": "Mframe-px/s", "ms_per_step": ms,
            "dtype": "fp32 storage, 3 x tf32 convs (VAE_FP32_TC; the parity mode VAE_FP32 runs on the CUDA cores)",
            "conv_tflops": tf, "conv_frac_of_3xtf32_peak": tf / eff_peak,
            "kernels": kernel_table(prof, args.steps, peaks)}


def run_ltx_encode(args, torch, vd, peaks, flush, stream):
    """The LTX-shaped encoder (the decoder read backwards): pixels [1,3,81,704,1280] -> moments
    [1,256,11,22,40], 1x4 patches; throughput in encoded Mframe-px/s of the input video."""
    cfg = synth.LTX_ENC
    params = synth.draw_params(cfg, 0)
    enc = vd.Encoder(cfg, params, vd.VAE_BF16)
    del params
    v = torch.from_numpy(synth.draw_video(cfg, 0)).cuda()
    out = torch.empty(enc.output_shape(v.shape), dtype=torch.float32, device="cuda")
    ms, prof = timed_decodes(torch, enc, lambda: enc.encode(v, out, 1, 4), args.steps, args.warmup, flush, stream)
    code, msg = enc.last_error()
    if code:
        raise RuntimeError(f"encode failed: {msg}")
    enc.close()
    fpx = v.shape[0] * v.shape[2] * v.shape[3] * v.shape[4]
    conv = conv_totals(prof)
    tf = conv["flops"] / (conv["ms"] / 1e3) / 1e12
    del v, out
    torch.cuda.empty_cache()
    return {"workload": f"ltx-shaped encoder, pixels {list(cfg.video_shape)} -> moments {list(cfg.latent_shape())}, "
                        "1x4 patches", "value": fpx / ms / 1e3, "unit": "encoded Mframe-px/s", "ms_per_step": ms,
            "conv_tflops": tf, "conv_frac_of_bf16_sustained": tf / peaks["bf16_tflops_sustained"],
            "kernels": kernel_table(prof, args.steps, peaks)}


def run_ltx(args, torch, vd, peaks, flush, stream):
    """The LTX-shaped 720p x 81f decode at 1x4 and 2x4 patches, and the batch-2 overlap-tiled LTX decode
    (latent [2,128,17,34,60] -> [2,3,129,1088,1920], 45 tiles of 8x16x16 latents, 1x4x4 overlap)."""
    res = {}
    for cfg, tiled in ((synth.LTX, False), (synth.LTX_TILED, True)):
        params = synth.draw_params(cfg, 0)
        dec = vd.Decoder(cfg, params, vd.VAE_BF16)
        del params
        z = torch.from_numpy(synth.draw_latent(cfg, 0)).cuda()
        out = torch.empty(dec.output_shape(z.shape), dtype=torch.bfloat16, device="cuda")
        runs = [("tiled", None)] if tiled else [("1x4", (1, 4)), ("2x4", (2, 4))]
        for tag, grid in runs:
            if tiled:
                tl = synth.LTX_TILING
                fn = lambda: dec.decode_tiled(z, tl.tile, tl.overlap, out)
            else:
                fn = lambda g=grid: dec.decode(z, out, g[0], g[1])
            ms, prof = timed_decodes(torch, dec, fn, args.steps, args.warmup, flush, stream)
            code, msg = vd.last_error(dec.h)
            if code:
                raise RuntimeError(f"{cfg.name} decode failed: {msg}")
            fpx = out.shape[0] * out.shape[2] * out.shape[3] * out.shape[4]
            conv = conv_totals(prof)
            tf = conv["flops"] / (conv["ms"] / 1e3) / 1e12
            res[f"{cfg.name}_{tag}"] = {
                "workload": f"{cfg.name}-shaped decoder, latent {list(cfg.latent_shape)} -> pixels {list(out.shape)}, "
                            + ("45 overlap tiles of 8x16x16 latents (1x4x4 overlap), blended" if tiled
                               else f"{grid[0]}x{grid[1]} spatial patches"),
                "value": fpx / ms / 1e3, "unit": "Mframe-px/s", "ms_per_step": ms,
                "conv_tflops": tf, "conv_frac_of_bf16_sustained": tf / peaks["bf16_tflops_sustained"],
                "kernels": kernel_table(prof, args.steps, peaks)}
        dec.close()
        del z, out
        torch.cuda.empty_cache()
    return res


def _time(torch, fn, steps, flush):
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    s = torch.cuda.current_stream()
    for a, b in evs:
        flush.zero_()
        a.record(s)
        fn()
        b.record(s)
    torch.cuda.synchronize()
    return sum(a.elapsed_time(b) for a, b in evs) / steps


def run_ops(args, torch, vd, peaks, flush):
    res = {}
    B, C, T, H, W = 1, 512, 21, 88, 160
    eh, ew = vd.patch_edges(H, 1), vd.patch_edges(W, 4)
    # (a) PatchGroupNorm + SiLU, 4 width patches
    x = torch.from_numpy(synth.draw_normal((B, T, H, W, C), 100)).to("cuda", torch.bfloat16)
    y = torch.empty_like(x)
    g = torch.ones(C, device="cuda")
    bt = torch.zeros(C, device="cuda")
    gd = vd.gn_desc(B, T, H, W, C, 32, eh, ew)
    ws = vd.gn_workspace(gd, "cuda")
    gn = vd.prepare_patch_groupnorm_silu(x, g, bt, y, ws, gd)  # arguments marshalled once
    ms = _time(torch, gn, args.steps, flush)
    nbytes = 3 * x.numel() * 2
    res["groupnorm_silu"] = {"workload": "[1,512,21,88,160] bf16, 32 groups, 4 width patches", "ms": ms,
                             "bytes": nbytes, "gbs": nbytes / ms / 1e6, "frac_of_hbm": nbytes / ms / 1e6 / peaks["hbm_gbs"],
                             "bound": "hbm"}
    # (a') channel RMS norm + SiLU on the same tensor (the Wan / LTX-2 norm family; no statistics pass)
    rms = vd.prepare_channel_rmsnorm_silu(x, g, bt, y, B, T, H, W, C)
    ms = _time(torch, rms, args.steps, flush)
    nbytes = 2 * x.numel() * 2
    res["channel_rmsnorm_silu"] = {"workload": "[1,512,21,88,160] bf16, per-pixel RMS over 512 channels", "ms": ms,
                                   "bytes": nbytes, "gbs": nbytes / ms / 1e6,
                                   "frac_of_hbm": nbytes / ms / 1e6 / peaks["hbm_gbs"], "bound": "hbm"}
    # (b) causal conv 3x3x3 512 -> 512, 4 width patches
    w = torch.from_numpy(synth.conv_weight(C, C, 101)).cuda()
    cd = vd.conv_desc(B, T, H, W, C, C, eh, ew)
    wp = vd.conv3d_pack_weights(w, cd)
    yc = torch.empty_like(x)
    ms = _time(torch, lambda: vd.conv3d_causal(x, wp, None, None, yc, cd), args.steps, flush)
    fl = 2.0 * 27 * C * C * T * H * W
    tr = _traffic("conv_tc_c2b")
    res["conv3d_causal"] = {"workload": "3x3x3 512->512 on [1,512,21,88,160] bf16, 4 width patches", "ms": ms,
                            "tflops": fl / ms / 1e9, "frac_of_bf16": fl / ms / 1e9 / peaks["bf16_tflops"],
                            "bound": "tensor", "traffic": tr["bytes_per_launch"] if tr else None}
    # (b') the same conv with e4m3 operands and per-channel-scaled e4m3 weights (kind::f8f6f4); the peak is
    # the measured bf16 peak x 2, the nominal dense fp8 : bf16 ratio (4.5 : 2.25 PFLOP/s)
    cd8 = vd.conv_desc(B, T, H, W, C, C, eh, ew, in_dtype=vd.VAE_FP8)
    wp8 = vd.conv3d_pack_weights(w, cd8)
    x8 = x.float().clamp(-448, 448).to(torch.float8_e4m3fn)  # input preparation, not timed
    ms = _time(torch, lambda: vd.conv3d_causal(x8, wp8, None, None, yc, cd8), args.steps, flush)
    res["conv3d_causal_fp8"] = {"workload": "3x3x3 512->512 on [1,512,21,88,160], e4m3 operands, bf16 out, 4 width patches",
                                "ms": ms, "tflops": fl / ms / 1e9, "frac_of_fp8": fl / ms / 1e9 / (2 * peaks["bf16_tflops"]),
                                "peak_kind": "fp8 dense = 2 x measured bf16 burst (nominal ratio)", "bound": "tensor",
                                "speedup_vs_bf16": res["conv3d_causal"]["ms"] / ms}
    del x, y, yc, wp, x8, wp8
    # (d) the pixel heads (conv_out + final depth-to-space, NCTHW pixels): Wan 256 -> 12, d2s (1,2,2) on
    # [1,256,81,352,640]; LTX 128 -> 48, d2s (1,4,4) on [1,128,81,176,320]; 4 width patches
    for name, Ci, Co, Hh, Wh, d2 in (("conv_head_wan", 256, 12, 352, 640, (1, 2, 2)),
                                     ("conv_head_ltx", 128, 48, 176, 320, (1, 4, 4))):
        Th = args.ops_frames or 81
        xh = torch.from_numpy(synth.draw_normal((1, Th, Hh, Wh, Ci), 102)).to("cuda", torch.bfloat16)
        wh = torch.from_numpy(synth.conv_weight(Co, Ci, 103)).cuda()
        hd = vd.conv_desc(1, Th, Hh, Wh, Ci, Co, vd.patch_edges(Hh, 1), vd.patch_edges(Wh, 4), d2s=d2, out_ncthw=True)
        whp = vd.conv3d_pack_weights(wh, hd)
        yh = torch.empty((1, Co // (d2[1] * d2[2]), Th, Hh * d2[1], Wh * d2[2]), dtype=torch.bfloat16, device="cuda")
        ms = _time(torch, lambda: vd.conv3d_causal(xh, whp, None, None, yh, hd), args.steps, flush)
        flh = 2.0 * 27 * Ci * Co * Th * Hh * Wh
        byh = xh.numel() * 2 + yh.numel() * 2
        t_floor = max(flh / (peaks["bf16_tflops"] * 1e12), byh / (peaks["hbm_gbs"] * 1e9)) * 1e3
        res[name] = {"workload": f"3x3x3 {Ci}->{Co}, d2s {d2}, on [1,{Ci},{Th},{Hh},{Wh}] bf16 -> NCTHW pixels, "
                                 "4 width patches", "ms": ms, "tflops": flh / ms / 1e9, "gbs": byh / ms / 1e6,
                     "roofline_ms": t_floor, "frac_of_roofline": t_floor / ms,
                     "bound": "max(FLOP / bf16 peak, bytes / HBM)"}
        del xh, yh, whp
    # (c) tile blend: 28 tiles of 256^2 with 64 px overlap -> [1, 3, 81, 704, 1280]
    meta = vd.tile_plan((81, 704, 1280), (81, 256, 256), (0, 64, 64), 1, 1, causal_t=False)
    tiles = [torch.from_numpy(synth.draw_normal((1, 3, m["pix"][1], m["pix"][3], m["pix"][5]), 200 + i)).to(
        "cuda", torch.bfloat16) for i, m in enumerate(meta)]
    outb = torch.empty((1, 3, 81, 704, 1280), dtype=torch.bfloat16, device="cuda")
    blend = vd.prepare_tile_blend(tiles, meta, outb)  # arguments marshalled once, outside the timing
    ms = _time(torch, blend, args.steps, flush)
    nbytes = sum(t.numel() for t in tiles) * 2 + outb.numel() * 2
    res["tile_blend"] = {"workload": f"{len(meta)} tiles of up to [1,3,81,256,256] bf16, 64 px overlap -> "
                                     "[1,3,81,704,1280]", "ms": ms, "bytes": nbytes, "gbs": nbytes / ms / 1e6,
                         "frac_of_hbm": nbytes / ms / 1e6 / peaks["hbm_gbs"], "bound": "hbm"}
    del tiles, outb, blend
    # (d) the blend of the batch-2 overlap-tiled LTX decode: 45 tiles overlapping in time and space
    cfg, tl = synth.LTX_TILED, synth.LTX_TILING
    if args.blend_small:  # a smaller case of the same plan for profiler captures: batch 1, 9 latent frames
        cfg = dataclasses.replace(cfg, latent_shape=(1, cfg.latent_shape[1], 9) + tuple(cfg.latent_shape[3:]))
    st, ss, _ = cfg.scale()
    meta = vd.tile_plan(cfg.latent_shape[2:], tl.tile, tl.overlap, st, ss)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(201)
    nbat = cfg.latent_shape[0]
    tiles = [torch.randn((nbat, 3, m["pix"][1], m["pix"][3], m["pix"][5]), generator=gen, device="cuda").to(
        torch.bfloat16) for m in meta]
    outb = torch.empty(cfg.output_shape(), dtype=torch.bfloat16, device="cuda")
    blend = vd.prepare_tile_blend(tiles, meta, outb)
    ms = _time(torch, blend, args.steps, flush)
    nbytes = sum(t.numel() for t in tiles) * 2 + outb.numel() * 2
    res["tile_blend_ltx_tiled"] = {"workload": f"{len(meta)} tiles of up to [{nbat},3,57,512,512] bf16 (overlap 8 frames, "
                                               f"128 px) -> {list(cfg.output_shape())}", "ms": ms, "bytes": nbytes,
                                   "gbs": nbytes / ms / 1e6, "frac_of_hbm": nbytes / ms / 1e6 / peaks["hbm_gbs"],
                                   "bound": "hbm"}
    del tiles, outb, blend
    return res


if __name__ == "__main__":
    main()
