#!/usr/bin/env python3
"""KDA hot-path benchmark: chunk-32 prefill + T=1 decode on GB300, one JSON line.

One step = one kda_prefill_ex call over the prefill workload followed by one kda_decode
call over the decode workload (both rows of the hot path), inputs resident in HBM.
Default workload: prefill 8 x 16384 tokens, H = 96, lower bound -8, FP32 initial states
N(0, 0.02), through kda_prefill_ex with its workspace (five full waves of one CTA per
chain, the 8 chains left over on the window schedule); decode H = 8, 4096 rows against a
16384-slot FP32 pool, scattered unique slots. L2 is flushed (a 512 MiB write) between
steps, outside the timed kernel segments. ``value`` is prefill tokens*heads/s over the
mean prefill time; decode rows*heads/s is reported beside it; ``roofline`` is the kernel
with the larger time share (the other kernel's roofline sits in its own object). The
small-B*H prefill (1 x 8192 tokens, H = 8, windowed) is timed after the main loop and
reported as ``prefill_small_bh``.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--prefill prefill_8x16384_h96|prefill_h8_t8192|prefill_varlen16_h32|prefill_h1_t64]
                  [--decode-rows R] [--state-dtype f32|bf16] [--no-e2e] [--no-cpu-baseline]

``--impl reference`` times the FP64 oracle (the CPU reference of this build) on the
host cores on a bounded sample of the same workload and prints the same JSON shape.
Each rank runs its own copy of the workload (weak scaling: chains are independent, so no
collective touches the data path); rank 0 prints the line with the maximum time over
ranks. ``--gpus N`` with N > 1 outside torchrun starts the N rank processes itself.
"""
from __future__ import annotations

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

METRIC = "KDA prefill tokens·heads/s (d=128) + decode rows·heads/s; % of roofline"
PREFILL_BYTES_PER_TOKEN_HEAD = 4 * 256 + 4 + 256  # q, k, v, g_raw (BF16 x 128) + beta + out
STATE_BYTES = 128 * 128 * 4                        # one FP32 state
PREFILL_FLOP_PER_TOKEN_HEAD = 6 * 128 * 128 + 8 * 32 * 128
DECODE_IO_BYTES_PER_ROW_HEAD = 4 * 256 + 4 + 256   # q, k, v, g_raw, beta, out
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--prefill", default="prefill_8x16384_h96")
    p.add_argument("--decode-rows", type=int, default=4096)
    p.add_argument("--state-dtype", default="f32", choices=["f32", "bf16"])
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-clocks", action="store_true")
    p.add_argument("--seqlens", default=None,
                   help="comma-separated sequence lengths replacing the prefill workload's (small ncu cases)")
    p.add_argument("--heads", type=int, default=None, help="head count replacing the prefill workload's")
    p.add_argument("--pool-slots", type=int, default=None, help="decode pool size replacing 16384 (small ncu cases)")
    p.add_argument("--decode-tokens", type=int, default=1,
                   help="tokens per decode row (kda_decode_ex, up to 16); above 1 the e2e and CPU legs are skipped")
    p.add_argument("--ckpt-every", type=int, default=0,
                   help="prefill also writes the FP32 state every N tokens (a multiple of 32) as checkpoints; "
                        "the e2e and CPU legs are then skipped")
    p.add_argument("--no-small-bh", action="store_true",
                   help="skip the secondary 1 x 8192 H8 windowed prefill measurement")
    p.add_argument("--no-sweep", action="store_true",
                   help="skip the decode sweep (rows 1 .. 4096, FP32 and BF16 pools) reported beside the line")
    p.add_argument("--decode-flags", default="",
                   help="decode input options for the timed decode: comma list of l2norm, beta_logits")
    p.add_argument("--no-windows", action="store_true",
                   help="run kda_prefill (sequential chunk loop) instead of kda_prefill_ex with a workspace")
    return p.parse_args(argv)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------------ distributed plumbing

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world, backend):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist if world > 1 else None


def max_over_ranks(value: float, dist, device=None) -> float:
    """The maximum of ``value`` over all ranks (identity on one rank)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def rank_seed(base: int, rank: int) -> int:
    """Each rank draws its own synthetic copy of the workload."""
    return base + 1000003 * rank


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """Samples the SM clock and the clock-event (throttle) reasons while the timed region runs.

    Reads NVML every 2 ms when libnvidia-ml loads (read-only queries: clock, maximum clock,
    event reasons), so that even a timed region of a few hundred milliseconds yields many
    samples; otherwise nvidia-smi every 100 ms. Nothing here changes a GPU setting."""

    SMI_FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                  "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                  "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    # NVML clock-event reason bits
    NVML_REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
                    0x40: "hw_thermal_slowdown"}
    NVML_CLOCK_SM = 1

    def __init__(self, index: int, pci_bus_id: str | None = None, period_s: float = 0.002):
        self.index, self.pci = index, pci_bus_id
        self.period = period_s
        self.proc = None
        self.thread = None
        self.lines = []
        self.samples = []  # (sm_mhz, reason bits)
        self.max_mhz = None
        self.source = None
        self._stop = threading.Event()

    # -- NVML through ctypes (the bindings package is not installed everywhere)
    def _nvml_open(self):
        import ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        handle = ctypes.c_void_p()
        rc = 1
        if self.pci:
            rc = lib.nvmlDeviceGetHandleByPciBusId_v2(self.pci.encode(), ctypes.byref(handle))
        if rc != 0:
            rc = lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.index), ctypes.byref(handle))
        if rc != 0:
            lib.nvmlShutdown()
            raise OSError("no NVML handle")
        reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons
        mx = ctypes.c_uint(0)
        if lib.nvmlDeviceGetMaxClockInfo(handle, self.NVML_CLOCK_SM, ctypes.byref(mx)) == 0:
            self.max_mhz = float(mx.value)
        return lib, handle, reasons

    def _nvml_loop(self, lib, handle, reasons):
        import ctypes
        mhz, bits = ctypes.c_uint(0), ctypes.c_ulonglong(0)
        try:
            while not self._stop.is_set():
                if (lib.nvmlDeviceGetClockInfo(handle, self.NVML_CLOCK_SM, ctypes.byref(mhz)) == 0 and
                        reasons(handle, ctypes.byref(bits)) == 0):
                    self.samples.append((float(mhz.value), int(bits.value)))
                self._stop.wait(self.period)
        finally:
            lib.nvmlShutdown()

    def __enter__(self):
        try:
            lib, handle, reasons = self._nvml_open()
            self.source = "nvml, every 2 ms"
            self.thread = threading.Thread(target=self._nvml_loop, args=(lib, handle, reasons), daemon=True)
            self.thread.start()
            return self
        except (OSError, AttributeError):
            pass
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.SMI_FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.source = "nvidia-smi, every 100 ms"
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        self._stop.set()
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=2)

    def summary(self):
        sm, reasons = [], set()
        smax = [self.max_mhz] if self.max_mhz else []
        for mhz, bits in self.samples:
            sm.append(mhz)
            reasons.update(name for bit, name in self.NVML_REASONS.items() if bits & bit)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for name, flag in zip(names, parts[4:8]):
                if flag.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "source": self.source}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax) if smax else None,
                "sm_min_mhz": min(sm), "reasons": sorted(reasons), "samples": len(sm), "source": self.source}


def pci_bus_id(device) -> str | None:
    """NVML's PCI bus id string of a torch CUDA device, when torch reports its PCI location."""
    import torch
    p = torch.cuda.get_device_properties(device)
    try:
        return f"{int(p.pci_domain_id):08X}:{int(p.pci_bus_id):02X}:{int(p.pci_device_id):02X}.0"
    except (AttributeError, TypeError, ValueError):
        return None


# ------------------------------------------------------------------ workloads

def prefill_workload(name, device, seed_offset=0, seqlens=None, heads=None):
    import dataclasses

    import kda_synth as S
    cfg = S.configs()[name]
    if seqlens or heads:
        cfg = dataclasses.replace(cfg, name=f"{name}[seqlens={seqlens or cfg.seqlens},heads={heads or cfg.num_heads}]",
                                  seqlens=list(seqlens or cfg.seqlens), num_heads=heads or cfg.num_heads)
    inp = S.prefill_inputs(cfg.seqlens, cfg.num_heads, seed=rank_seed(cfg.seed, seed_offset), init_std=cfg.init_std,
                           device=device)
    return cfg, inp


def decode_workload(rows, state_dtype, device, seed_offset=0, pool_slots=None, tokens=1):
    import dataclasses

    import kda_synth as S
    cfg = S.configs()["decode_h8_pool16384"]
    if pool_slots:
        cfg = dataclasses.replace(cfg, num_slots=pool_slots)
    seed = rank_seed(cfg.seed, seed_offset)
    pool = S.state_pool(cfg.num_slots, cfg.num_heads, state_dtype, std=cfg.pool_std, seed=seed, device=device)
    inp = S.decode_inputs(rows * tokens, cfg.num_heads, seed=seed, device=device)
    if tokens > 1:  # [rows, tokens, H, 128] and [rows, tokens, H]
        inp = {k: v.view(rows, tokens, *v.shape[1:]) for k, v in inp.items()}
    inp["slot_idx"] = S.slot_indices(rows, cfg.num_slots, seed=seed, device=device)
    return cfg, pool, inp


def prefill_units(cfg):
    return cfg.total_tokens * cfg.num_heads


def prefill_bytes(cfg):
    chains = len(cfg.seqlens) * cfg.num_heads
    state_io = chains * STATE_BYTES * (2 if cfg.init_std is not None else 1)
    return prefill_units(cfg) * PREFILL_BYTES_PER_TOKEN_HEAD + state_io


def decode_bytes(rows, heads, state_dtype, tokens=1):
    per_state = 128 * 128 * (4 if state_dtype == "f32" else 2)
    return rows * heads * (2 * per_state + tokens * DECODE_IO_BYTES_PER_ROW_HEAD) + rows * 4


# ------------------------------------------------------------------ our arm

def ms_stats(values):
    """mean, median and minimum of per-step milliseconds."""
    return {"mean": sum(values) / len(values), "median": statistics.median(values), "min": min(values)}


def prefill_roofline(pcfg, ms, peaks, peak_src, traffic, kernel, extra_bytes=0):
    """HBM roofline of a prefill schedule over its event time, with the tensor fraction beside it."""
    p_bytes = prefill_bytes(pcfg) + extra_bytes
    gbs = p_bytes / (ms * 1e-3) / 1e9
    flop = prefill_units(pcfg) * PREFILL_FLOP_PER_TOKEN_HEAD
    tflops = flop / (ms * 1e-3) / 1e12
    roof = {"bound": "hbm", "achieved": round(gbs, 2), "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": round(gbs / peaks["hbm_gbs"], 5), "traffic": traffic, "kernel": kernel, "peak_source": peak_src,
            "algorithmic_bytes_per_launch": p_bytes,
            "tensor": {"achieved": round(tflops, 3), "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                       "frac": round(tflops / peaks["bf16_tflops"], 5), "flop_per_launch": flop}}
    if traffic:
        roof["frac_of_traffic"] = round(traffic / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 5)
    return roof


def prefill_schedule(K, pcfg, device, no_windows):
    """The workspace kda_prefill_ex uses for this workload (None: sequential), the number of
    chains in full waves ahead of a windowed tail, and the number of launches per call."""
    import torch
    ws = None if no_windows else K.prefill_workspace(len(pcfg.seqlens), pcfg.total_tokens, pcfg.num_heads, device)
    chains = len(pcfg.seqlens) * pcfg.num_heads
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    full_waves = chains // sms if ws is not None else 0
    # chunk loop (full waves and window 0) + window pass + carry + output pass, or the chunk loop
    return ws, full_waves, (4 if ws is not None else 1)


def schedule_name(ws, full_waves, chains, sms):
    if ws is None:
        return "sequential chunk loop"
    head = (f"{full_waves} full waves of the chunk loop, then {chains - full_waves * sms} chains on "
            if full_waves else "")
    return head + f"windows ({ws.numel() >> 20} MiB workspace)"


def prefill_traffic(traffic, pcfg, ws, full_waves):
    """ncu DRAM bytes of one prefill call, scaled from the captured case by units processed: the
    sequential chunk-loop record for the sequential schedule; for the window schedule the record
    of the same schedule (all four launches), with or without full waves ahead of it."""
    units = prefill_units(pcfg)
    if ws is None:
        return scaled_traffic(traffic, "kda_prefill_tc_kernel", units)
    key = "prefill_window_schedule_tail" if full_waves else "prefill_window_schedule_small_bh"
    return scaled_traffic(traffic, key, units, len(pcfg.seqlens) * pcfg.num_heads)


def run_ours(args):
    import torch

    import kda_recurrent_gb300 as K

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist = init_dist(world, "nccl")
    K.load(build_if_missing=True)
    peaks, peak_src = load_peaks()

    seqlens = [int(x) for x in args.seqlens.split(",")] if args.seqlens else None
    pcfg, pin = prefill_workload(args.prefill, device, rank, seqlens, args.heads)
    T = args.decode_tokens
    if not 1 <= T <= 16:
        raise SystemExit("--decode-tokens takes 1 .. 16")
    if T > 1 or args.ckpt_every:  # the e2e and CPU legs time the plain calls
        args.no_e2e = args.no_cpu_baseline = True
    dcfg, pool, din = decode_workload(args.decode_rows, args.state_dtype, device, rank, args.pool_slots, T)
    scale = pcfg.scale
    out = torch.empty_like(pin["q"])
    fin = torch.empty(len(pcfg.seqlens), pcfg.num_heads, 128, 128, dtype=torch.float32, device=device)
    dout = torch.empty_like(din["q"])
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    flush = torch.empty(max(2 * l2, 512 << 20), dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    ws, full_waves, prefill_launches = prefill_schedule(K, pcfg, device, args.no_windows)
    chains = len(pcfg.seqlens) * pcfg.num_heads

    ck = ck_off = None
    ck_rows = 0
    if args.ckpt_every:
        if args.ckpt_every % 32:
            raise SystemExit("--ckpt-every takes a multiple of 32")
        per_seq = [n // args.ckpt_every for n in pcfg.seqlens]
        ck_rows = sum(per_seq)
        ck = torch.empty(max(ck_rows, 1), pcfg.num_heads, 128, 128, dtype=torch.float32, device=device)
        ck_off = torch.tensor([sum(per_seq[:i]) for i in range(len(per_seq))], dtype=torch.int32, device=device)

    def prefill_call():
        K.kda_prefill_ex(pin["q"], pin["k"], pin["v"], pin["g_raw"], pin["beta"], pin["cu_seqlens"],
                         pin["init_state"], out, fin, scale, pcfg.lower_bound, pcfg.gate_mode, ws, stream,
                         checkpoints=ck, ckpt_offsets=ck_off, ckpt_every=args.ckpt_every)

    dflags = decode_flags(args.decode_flags)
    if dflags:  # the e2e and CPU legs time the plain calls
        args.no_e2e = args.no_cpu_baseline = True

    def decode_call():
        if T == 1 and not dflags:
            K.kda_decode(din["q"], din["k"], din["v"], din["g_raw"], din["beta"], din["slot_idx"], pool, dout,
                         dcfg.scale, dcfg.lower_bound, dcfg.gate_mode, stream)
        else:
            K.kda_decode_ex(din["q"], din["k"], din["v"], din["g_raw"], din["beta"], din["slot_idx"], pool, dout,
                            dcfg.scale, dcfg.lower_bound, dcfg.gate_mode, flags=dflags, norm_eps=1e-6,
                            stream=stream)

    for _ in range(args.warmup):
        flush.zero_()
        prefill_call()
        decode_call()
    torch.cuda.synchronize(device)
    st, detail = K.kda_device_status()
    if st != K.KDA_OK:
        raise RuntimeError(f"device status {st} ({detail}) after warm-up")

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(device)
    sampler = ClockSampler(local, pci_bus_id(device)) if not args.no_clocks else None
    if sampler:
        sampler.__enter__()
    t_wall = time.perf_counter()
    for s in range(args.steps):
        flush.zero_()
        ev[s][0].record(stream)
        prefill_call()
        ev[s][1].record(stream)
        decode_call()
        ev[s][2].record(stream)
    torch.cuda.synchronize(device)
    wall = time.perf_counter() - t_wall
    if sampler:
        sampler.__exit__(None, None, None)
    if dist is not None:
        dist.barrier()
    p_st = ms_stats([ev[s][0].elapsed_time(ev[s][1]) for s in range(args.steps)])
    d_st = ms_stats([ev[s][1].elapsed_time(ev[s][2]) for s in range(args.steps)])
    # the slowest rank sets the time of the job
    p_st = {k: max_over_ranks(v, dist, device) for k, v in p_st.items()}
    d_st = {k: max_over_ranks(v, dist, device) for k, v in d_st.items()}
    p_mean, d_mean = p_st["mean"], d_st["mean"]
    st, detail = K.kda_device_status()
    if st != K.KDA_OK:
        raise RuntimeError(f"device status {st} ({detail}) after the timed region")
    traffic = load_traffic()

    small = None
    if not args.no_small_bh and not args.seqlens and not args.heads and args.prefill != "prefill_h8_t8192":
        small = measure_small_bh(K, args, device, rank, flush, stream, dist, peaks, peak_src, traffic, sms)
    sweep = None
    if not args.no_sweep and not args.pool_slots and T == 1 and not dflags:
        sweep = measure_decode_sweep(K, args, device, rank, flush, stream, dist, peaks, pool)

    e2e = None if args.no_e2e else measure_e2e(K, pcfg, pin, dcfg, din, pool, stream, device, args, dist, ws)
    cpu = None
    if not args.no_cpu_baseline and rank == 0 and world == 1:
        cpu = cpu_baseline(pcfg, pin, dcfg, din, pool)
    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return None

    p_units = prefill_units(pcfg) * world
    d_units = args.decode_rows * dcfg.num_heads * T * world  # (row, head) items x tokens
    p_rate = p_units / (p_mean * 1e-3)
    d_rate = d_units / (d_mean * 1e-3)
    d_bytes = decode_bytes(args.decode_rows, dcfg.num_heads, args.state_dtype, T)
    d_gbs = d_bytes / (d_mean * 1e-3) / 1e9
    waves = math.ceil(chains / sms)  # one CTA per chain, one CTA per SM
    p_kernel = ("kda_prefill_tc_kernel (sequential chunk loop)" if ws is None else
                ("kda_prefill_tc_kernel full waves + " if full_waves else "") +
                "window schedule of the tail (window 0, window pass, carry, output pass)")
    prefill_roof = prefill_roofline(pcfg, p_mean, peaks, peak_src,
                                    prefill_traffic(traffic, pcfg, ws, full_waves) if not ck_rows else None, p_kernel,
                                    extra_bytes=ck_rows * pcfg.num_heads * STATE_BYTES)
    d_kernel = (decode_kernel_name(args.decode_rows * dcfg.num_heads, sms, args.state_dtype) if T == 1
                else "kda_decode_stream_kernel")
    d_traffic = (scaled_traffic(traffic, f"{d_kernel}<{args.state_dtype}>", args.decode_rows * dcfg.num_heads)
                 if T == 1 else None)
    decode_roof = {"bound": "hbm", "achieved": round(d_gbs, 2), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                   "frac": round(d_gbs / peaks["hbm_gbs"], 5), "traffic": d_traffic,
                   "kernel": d_kernel, "peak_source": peak_src, "algorithmic_bytes_per_launch": d_bytes}
    if d_traffic:
        decode_roof["frac_of_traffic"] = round(d_traffic / (d_mean * 1e-3) / 1e9 / peaks["hbm_gbs"], 5)
        if d_traffic < d_bytes:
            decode_roof["note"] = ("algorithmic bytes exceed the DRAM traffic ncu counts: the last state "
                                   "writes are still in L2 when the kernel ends, so frac can pass 1.0; "
                                   "frac_of_traffic is the DRAM-side fraction")
    dominant = prefill_roof if p_mean >= d_mean else decode_roof
    line = {
        "metric": METRIC, "value": round(p_rate, 1), "unit": "tokens*heads/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(p_mean + d_mean, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": f"{pcfg.name} + decode_h8_rows{args.decode_rows}_{args.state_dtype}_pool{dcfg.num_slots}",
                   "prefill": {"seqlens": pcfg.seqlens if len(set(pcfg.seqlens)) > 1 and len(pcfg.seqlens) <= 16
                               else f"{len(pcfg.seqlens)} x {pcfg.seqlens[0]}" if len(set(pcfg.seqlens)) == 1
                               else f"{len(pcfg.seqlens)} seqs",
                               "heads": pcfg.num_heads, "gate": pcfg.gate_mode, "lower_bound": pcfg.lower_bound,
                               "init_state": pcfg.init_std is not None, "ckpt_every": args.ckpt_every},
                   "decode": {"rows": args.decode_rows, "heads": dcfg.num_heads, "pool_slots": dcfg.num_slots,
                              "state_dtype": args.state_dtype, "tokens_per_row": T,
                              "options": args.decode_flags or "none"},
                   "precision": "bf16 operands, tf32 state update, fp32 state and accumulation",
                   "prefill_schedule": schedule_name(ws, full_waves, chains, sms),
                   "l2": f"flushed between steps ({flush.numel() >> 20} MiB write)",
                   "parallelism": f"replicas{world}" if world > 1 else "single"},
        "prefill": {"value": round(p_rate, 1), "unit": "tokens*heads/s", "ms": round(p_mean, 4),
                    "ms_median": round(p_st["median"], 4), "ms_min": round(p_st["min"], 4),
                    "value_at_median": round(p_units / (p_st["median"] * 1e-3), 1),
                    "us_per_chunk_per_chain": round(p_mean * 1e3 / (math.ceil(max(pcfg.seqlens) / 32) * waves), 4),
                    "waves": waves},
        "decode": {"value": round(d_rate, 1), "unit": "rows*heads/s" if T == 1 else "tokens*heads/s",
                   "ms": round(d_mean, 4), "ms_median": round(d_st["median"], 4), "ms_min": round(d_st["min"], 4),
                   "roofline": decode_roof},
        "roofline": dominant,
        "roofline_prefill": prefill_roof,
        "gpu_launches": (prefill_launches + 1) * args.steps,
        "wall_s_timed_region": round(wall, 4),
    }
    if small is not None:
        line["prefill_small_bh"] = small
    if sweep is not None:
        line["decode_sweep"] = sweep
    if sampler:
        line["clocks"] = sampler.summary()
    if e2e is not None:
        line["e2e"] = e2e
    if cpu is not None:
        line["cpu_baseline"] = cpu
    if dist is not None:
        dist.destroy_process_group()
    return line


def decode_flags(text):
    """KDA_DECODE_* bits from a comma list of option names."""
    names = {"l2norm": 1, "beta_logits": 2}
    bits = 0
    for name in filter(None, (x.strip() for x in text.split(","))):
        if name not in names:
            raise SystemExit(f"--decode-flags: unknown option {name!r} (l2norm, beta_logits)")
        bits |= names[name]
    return bits


def measure_decode_sweep(K, args, device, rank, flush, stream, dist, peaks, pool_f32):
    """The whole decode workload: rows 1, 2, 4 .. 4096 x H8 on 16384-slot FP32 and BF16 pools,
    each row count timed over --steps calls (L2 flushed between them). Reports per row count the
    median time in microseconds and the fraction of HBM bandwidth on the state and token bytes."""
    import torch

    import kda_synth as S
    cfg = S.configs()["decode_h8_pool16384"]
    H = cfg.num_heads
    res = {}
    for dt in ("f32", "bf16"):
        pool = pool_f32 if (dt == "f32" and args.state_dtype == "f32") else \
            S.state_pool(cfg.num_slots, H, dt, std=cfg.pool_std, seed=rank_seed(cfg.seed, rank), device=device)
        us, frac = [], []
        for rows in cfg.rows:
            d = S.decode_inputs(rows, H, seed=rank_seed(cfg.seed, rank) + rows, device=device)
            slots = S.slot_indices(rows, cfg.num_slots, seed=rank_seed(cfg.seed, rank), device=device)
            out = torch.empty_like(d["q"])

            def call():
                K.kda_decode(d["q"], d["k"], d["v"], d["g_raw"], d["beta"], slots, pool, out, cfg.scale,
                             cfg.lower_bound, cfg.gate_mode, stream)

            for _ in range(2):
                call()
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(args.steps)]
            for a_, b_ in ev:
                flush.zero_()
                a_.record(stream)
                call()
                b_.record(stream)
            torch.cuda.synchronize(device)
            ms = max_over_ranks(statistics.median(a_.elapsed_time(b_) for a_, b_ in ev), dist, device)
            us.append(round(ms * 1e3, 2))
            frac.append(round(decode_bytes(rows, H, dt) / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4))
        res[dt] = {"us_median": us, "hbm_frac": frac}
        if pool is not pool_f32:
            del pool
    st, detail = K.kda_device_status()
    if st != K.KDA_OK:
        raise RuntimeError(f"device status {st} ({detail}) after the decode sweep")
    return {"rows": list(cfg.rows), "heads": H, "pool_slots": cfg.num_slots, **res,
            "timing": "CUDA events per call, L2 flushed between calls, median of --steps calls"}


def measure_small_bh(K, args, device, rank, flush, stream, dist, peaks, peak_src, traffic, sms):
    """The small-B*H prefill (1 x 8192 tokens, H8: 8 chains on the window schedule), timed over
    --steps calls with L2 flushed between them; reported beside the main line."""
    import torch
    cfg, inp = prefill_workload("prefill_h8_t8192", device, rank)
    ws, full_waves, launches = prefill_schedule(K, cfg, device, args.no_windows)
    out = torch.empty_like(inp["q"])
    fin = torch.empty(1, cfg.num_heads, 128, 128, dtype=torch.float32, device=device)

    def call():
        K.kda_prefill_ex(inp["q"], inp["k"], inp["v"], inp["g_raw"], inp["beta"], inp["cu_seqlens"],
                         inp["init_state"], out, fin, cfg.scale, cfg.lower_bound, cfg.gate_mode, ws, stream)

    for _ in range(args.warmup):
        flush.zero_()
        call()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    torch.cuda.synchronize(device)
    for s in range(args.steps):
        flush.zero_()
        ev[s][0].record(stream)
        call()
        ev[s][1].record(stream)
    torch.cuda.synchronize(device)
    st = ms_stats([a.elapsed_time(b) for a, b in ev])
    st = {k: max_over_ranks(v, dist, device) for k, v in st.items()}
    units = prefill_units(cfg)
    world = dist.get_world_size() if dist is not None else 1
    return {"workload": cfg.name, "value": round(units * world / (st["mean"] * 1e-3), 1), "unit": "tokens*heads/s",
            "ms": round(st["mean"], 4), "ms_median": round(st["median"], 4), "ms_min": round(st["min"], 4),
            "us_per_chunk_per_chain": round(st["mean"] * 1e3 / math.ceil(max(cfg.seqlens) / 32), 4),
            "schedule": schedule_name(ws, full_waves, len(cfg.seqlens) * cfg.num_heads, sms),
            "gpu_launches": launches * args.steps,
            "roofline": prefill_roofline(cfg, st["mean"], peaks, peak_src, prefill_traffic(traffic, cfg, ws, full_waves),
                                         "window schedule (window 0, window pass, carry, output pass)"
                                         if ws is not None else "kda_prefill_tc_kernel (sequential chunk loop)")}


def measure_e2e(K, pcfg, pin, dcfg, din, pool, stream, device, args, dist, ws):
    """Same metric through the C ABI from pinned host buffers, every step's inputs copied in
    and its results (prefill out + final state, decode out) copied back inside the timed
    region. Steps are pipelined over three streams, as a serving loop would run them: the
    H2D copy of step s+1 and the D2H copy of step s-1 overlap the kernels of step s, with
    two device copies of every input and output."""
    import torch
    host_p = {k: (v.to("cpu").pin_memory() if v is not None else None) for k, v in pin.items()}
    host_d = {k: v.to("cpu").pin_memory() for k, v in din.items()}
    dev_p = [{k: (torch.empty_like(v, device=device) if v is not None else None) for k, v in host_p.items()}
             for _ in range(2)]
    dev_d = [{k: torch.empty_like(v, device=device) for k, v in host_d.items()} for _ in range(2)]
    out = [torch.empty_like(dev_p[0]["q"]) for _ in range(2)]
    fin = [torch.empty(len(pcfg.seqlens), pcfg.num_heads, 128, 128, dtype=torch.float32, device=device)
           for _ in range(2)]
    dout = [torch.empty_like(dev_d[0]["q"]) for _ in range(2)]
    h_out = [torch.empty(out[0].shape, dtype=out[0].dtype).pin_memory() for _ in range(2)]
    h_fin = [torch.empty(fin[0].shape, dtype=fin[0].dtype).pin_memory() for _ in range(2)]
    h_dout = [torch.empty(dout[0].shape, dtype=dout[0].dtype).pin_memory() for _ in range(2)]
    h2d = sum(v.numel() * v.element_size() for v in host_p.values() if v is not None)
    h2d_d = sum(v.numel() * v.element_size() for v in host_d.values())
    d2h = h_out[0].numel() * 2 + h_fin[0].numel() * 4
    d2h_d = h_dout[0].numel() * 2
    s_in, s_out = torch.cuda.Stream(device), torch.cuda.Stream(device)

    def pipeline(nsteps, copy_in, compute, copy_out):
        """Runs nsteps pipelined steps; returns the CUDA-event time from the first copy in to
        the last copy out, in ms."""
        ev = lambda: torch.cuda.Event(enable_timing=False)
        in_done, comp_done, out_done = [ev() for _ in range(nsteps)], [ev() for _ in range(nsteps)], [ev() for _ in range(nsteps)]
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(s_in)
        for i in range(nsteps):
            b = i & 1
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(comp_done[i - 2])  # buffer b's inputs are read
                copy_in(b)
                in_done[i].record(s_in)
            stream.wait_event(in_done[i])
            if i >= 2:
                stream.wait_event(out_done[i - 2])  # buffer b's outputs are copied out
            compute(b)
            comp_done[i].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(comp_done[i])
                copy_out(b)
                out_done[i].record(s_out)
        t1.record(s_out)
        torch.cuda.synchronize(device)
        return t0.elapsed_time(t1)

    def p_in(b):
        for k2, v in host_p.items():
            if v is not None:
                dev_p[b][k2].copy_(v, non_blocking=True)

    def p_comp(b):
        d = dev_p[b]
        K.kda_prefill_ex(d["q"], d["k"], d["v"], d["g_raw"], d["beta"], d["cu_seqlens"], d["init_state"], out[b],
                         fin[b], pcfg.scale, pcfg.lower_bound, pcfg.gate_mode, ws, stream)

    def p_out(b):
        h_out[b].copy_(out[b], non_blocking=True)
        h_fin[b].copy_(fin[b], non_blocking=True)

    def d_in(b):
        for k2, v in host_d.items():
            dev_d[b][k2].copy_(v, non_blocking=True)

    def d_comp(b):
        d = dev_d[b]
        K.kda_decode(d["q"], d["k"], d["v"], d["g_raw"], d["beta"], d["slot_idx"], pool, dout[b], dcfg.scale,
                     dcfg.lower_bound, dcfg.gate_mode, stream)

    def d_out(b):
        h_dout[b].copy_(dout[b], non_blocking=True)

    steps = max(3, args.steps // 2)
    pipeline(max(2, args.warmup), p_in, p_comp, p_out)  # warm-up
    p_ms = max_over_ranks(pipeline(steps, p_in, p_comp, p_out) / steps, dist, device)
    pipeline(max(2, args.warmup), d_in, d_comp, d_out)
    d_ms = max_over_ranks(pipeline(steps, d_in, d_comp, d_out) / steps, dist, device)
    world = dist.get_world_size() if dist is not None else 1
    return {"value": round(prefill_units(pcfg) * world / (p_ms * 1e-3), 1), "unit": "tokens*heads/s",
            "h2d_bytes_per_step": int(h2d + h2d_d), "d2h_bytes_per_step": int(d2h + d2h_d),
            "prefill_ms": round(p_ms, 4), "decode_ms": round(d_ms, 4),
            "decode_value": round(args.decode_rows * dcfg.num_heads * world / (d_ms * 1e-3), 1),
            "decode_unit": "rows*heads/s", "schedule": "H2D, kernels and D2H of consecutive steps overlap "
            "on three streams; two device copies of inputs and outputs"}


def decode_kernel_name(items: int, sms: int, state_dtype: str = "f32") -> str:
    """The decode kernel the library launches for one token per row: the streaming
    schedule from 4 (FP32 states) or 3 (BF16) (row, head) items per SM on, the register
    schedule below that."""
    return "kda_decode_stream_kernel" if items >= (4 if state_dtype == "f32" else 3) * sms else "kda_decode_kernel"


def source_digest(kernel_file: str) -> str:
    import hashlib
    with open(os.path.join(ROOT, "kda_recurrent_gb300", "csrc", kernel_file), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def load_traffic():
    """Per-unit DRAM bytes of each kernel from the committed ncu summary (profiles/traffic.json),
    kept only while the kernel source still has the digest the counters were taken on."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return {}
    out = {}
    for name, rec in d.items():
        try:
            if source_digest(rec["source"]) == rec["source_sha256_16"]:
                out[name] = rec
        except (OSError, KeyError):
            continue
    return out


def scaled_traffic(traffic, kernel, units, chains=0):
    """ncu DRAM bytes per launch, scaled from the captured case to this launch by units processed
    (plus, where the record separates it, the state traffic of each chain)."""
    rec = traffic.get(kernel)
    if rec is None:
        return None
    return int(rec["dram_bytes_per_unit"] * units + rec.get("dram_bytes_per_chain", 0) * chains)


# ------------------------------------------------------------------ oracle timing (CPU baseline)

def oracle_sample(pcfg, pin, dcfg, din, pool, budget_s=20.0):
    """Times the FP64 oracle on the host cores on bounded samples of the workload."""
    import torch

    import oracle
    H = pcfg.num_heads
    cu = pin["cu_seqlens"].tolist()
    # only the first sequence is ever sampled: copy just its tokens to the host
    cpu_p = {k: pin[k][cu[0]:cu[1]].to("cpu") for k in ("q", "k", "v", "g_raw", "beta")}
    cpu_p["init_state"] = None if pin["init_state"] is None else pin["init_state"][:1].to("cpu")
    # prefill sample: every head of the first sequence, first `toks` tokens (grown to fill the budget)
    toks = min(512, cu[1] - cu[0])
    res = {}
    while True:
        sub = {k: cpu_p[k][:toks] for k in ("q", "k", "v", "g_raw", "beta")}
        init = cpu_p["init_state"]
        t0 = time.perf_counter()
        _, _, threads = oracle.prefill(sub["q"], sub["k"], sub["v"], sub["g_raw"], sub["beta"],
                                       torch.tensor([0, toks], dtype=torch.int32), init, scale=pcfg.scale,
                                       lower_bound=pcfg.lower_bound, gate_mode=pcfg.gate_mode)
        dt = time.perf_counter() - t0
        res["prefill"] = (toks * H / dt, threads, f"sequence 0, first {toks} tokens, all {H} heads")
        if dt > budget_s / 4 or toks >= cu[1] - cu[0]:
            break
        toks = min(cu[1] - cu[0], toks * 4)
    rows = min(din["q"].shape[0], 1024)
    gathered = pool[din["slot_idx"][:rows].long()].to("cpu")
    t0 = time.perf_counter()
    _, _, threads_d = oracle.decode(din["q"][:rows].cpu(), din["k"][:rows].cpu(), din["v"][:rows].cpu(),
                                    din["g_raw"][:rows].cpu(), din["beta"][:rows].cpu(), gathered, scale=dcfg.scale,
                                    lower_bound=dcfg.lower_bound, gate_mode=dcfg.gate_mode)
    dt = time.perf_counter() - t0
    res["decode"] = (rows * dcfg.num_heads / dt, threads_d, f"first {rows} rows, all {dcfg.num_heads} heads")
    return res


def cpu_baseline(pcfg, pin, dcfg, din, pool):
    res = oracle_sample(pcfg, pin, dcfg, din, pool)
    p_rate, p_threads, p_sample = res["prefill"]
    d_rate, d_threads, d_sample = res["decode"]
    return {"value": round(p_rate, 2), "unit": "tokens*heads/s", "cores": p_threads, "kind": "oracle",
            "sample": f"prefill: {p_sample}", "host_cores": os.cpu_count(),
            "decode": {"value": round(d_rate, 2), "unit": "rows*heads/s", "cores": d_threads, "sample": d_sample}}


# ------------------------------------------------------------------ reference arm (the oracle)

def run_reference(args):
    world, rank, _ = dist_env()
    if world > 1 and rank != 0:
        return None
    import torch

    import kda_synth as S
    # the oracle samples only the first sequence, so only that sequence is drawn on the host
    first = S.configs()[args.prefill].seqlens[:1]
    pcfg, pin = prefill_workload(args.prefill, "cpu", 0, seqlens=first)
    dcfg = S.configs()["decode_h8_pool16384"]
    din = S.decode_inputs(min(args.decode_rows, 1024), dcfg.num_heads, seed=dcfg.seed)
    din["slot_idx"] = torch.arange(din["q"].shape[0], dtype=torch.int32)
    pool = S.state_pool(din["q"].shape[0], dcfg.num_heads, args.state_dtype, std=dcfg.pool_std, seed=dcfg.seed)
    budget = max(4.0, 150.0 / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        oracle_sample(pcfg, pin, dcfg, din, pool, budget_s=budget)
    p_rates, d_rates = [], []
    t0 = time.perf_counter()
    for _ in range(args.steps):
        r = oracle_sample(pcfg, pin, dcfg, din, pool, budget_s=budget)
        p_rates.append(r["prefill"][0])
        d_rates.append(r["decode"][0])
    wall = time.perf_counter() - t0
    p_rate = statistics.median(p_rates)
    return {"impl": "reference", "metric": METRIC, "value": round(p_rate, 2), "unit": "tokens*heads/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(wall * 1e3 / max(1, args.steps), 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"{args.prefill} + decode_h8_rows{args.decode_rows}_{args.state_dtype}_pool{dcfg.num_slots}",
                       "note": "FP64 CPU oracle on bounded samples of the workload (prefill: a prefix of "
                               "sequence 0, all heads; decode: the first rows)"},
            "decode": {"value": round(statistics.median(d_rates), 2), "unit": "rows*heads/s"},
            "cpu_baseline": {"value": round(p_rate, 2), "unit": "tokens*heads/s", "cores": r["prefill"][1],
                             "kind": "oracle", "sample": f"prefill: {r['prefill'][2]}; decode: {r['decode'][2]}"},
            "e2e": {"value": round(p_rate, 2), "unit": "tokens*heads/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def free_port() -> int:
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def launch_replicas(n: int, argv, cmd=None, timeout_s=None) -> int:
    """Starts ranks 0 .. n-1 of this benchmark as child processes on one node (one per GPU), with
    WORLD_SIZE / RANK / LOCAL_RANK and a 127.0.0.1 rendezvous in their environment, as torchrun
    would; rank 0 prints the JSON line. If a rank fails, the others are stopped. Returns the
    first non-zero exit code, else 0."""
    port = free_port()
    cmd = cmd or [sys.executable, os.path.abspath(__file__), *argv]
    procs = []
    for r in range(n):
        env = dict(os.environ, WORLD_SIZE=str(n), RANK=str(r), LOCAL_RANK=str(r), LOCAL_WORLD_SIZE=str(n),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        procs.append(subprocess.Popen(cmd, env=env))
    t0 = time.monotonic()
    rc = 0
    while [p.poll() for p in procs].count(None):  # polls every rank, so each exit code is seen
        failed = [p.returncode for p in procs if p.returncode not in (None, 0)]
        late = timeout_s is not None and time.monotonic() - t0 > timeout_s
        if failed or late:
            rc = failed[0] if failed else 124
            for p in procs:
                if p.poll() is None:
                    p.terminate()
            for p in procs:
                try:
                    p.wait(timeout=30)
                except subprocess.TimeoutExpired:
                    p.kill()
            break
        time.sleep(0.05)
    for p in procs:
        if rc == 0 and p.returncode:
            rc = p.returncode
    return rc


def main(argv=None):
    argv = sys.argv[1:] if argv is None else list(argv)
    args = parse_args(argv)
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        sys.exit(launch_replicas(args.gpus, argv))
    line = run_reference(args) if args.impl == "reference" else run_ours(args)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
