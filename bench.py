"""Steady-state serving benchmark of the autoregressive-denoising DiT wave path.

One step = one wave: every ready (chunk, step) task of every stream through
in-proj, all B blocks (LN1+mod, QKV+RoPE+KV append, window attention,
out-proj+gated residual, LN2+mod, up+GELU, down+gated residual) and the
final adaLN + velocity head + Euler update.  In a steady wave (every task at
a full KV window) each stream emits one chunk, so ms/step = per-stream
ms/chunk and value = aggregate chunks/s.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME]
  python bench.py --impl reference ...   # the CPU oracle on the host cores

N > 1 (under torchrun): independent replicas, one per GPU (the path has no
exchange step); value = chunks of all ranks / max-over-ranks time.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402

METRIC = "steady-state ms/chunk & chunks/s on 1 GB300; tensor-pipe % of BF16 peak"
# every model configuration, measured after the headline one in the default run
SWEEP = ["tiny", "wan21_1p3b", "wan22_5b", "wan21_1p3b_x8", "wan21_14b"]
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def workload_name(cfg_name: str, cfg: dict) -> str:
    return (f"{cfg_name}: {cfg['B']} blocks x {cfg['S']} steps, d={cfg['d']}, "
            f"{cfg['H']}x{cfg['dh']} heads, F={cfg['F']}, C={cfg['C']}, T={cfg['T']}, "
            f"W={cfg['W']}, {cfg['n_streams']} stream(s) x {cfg['n_chunks']} chunks")


def wave_flops(cfg: dict) -> float:
    """Algorithmic FLOPs of one steady wave (every task at a full window)."""
    n_task = cfg["S"] * cfg["n_streams"]
    M = n_task * cfg["T"]
    d, F, B, C, T = cfg["d"], cfg["F"], cfg["B"], cfg["C"], cfg["T"]
    Lk = (cfg["W"] + 1) * T
    gemm = 2.0 * M * B * (4 * d * d + 2 * d * F)
    attn = 4.0 * T * Lk * d * n_task * B
    io = 4.0 * M * C * d
    return gemm + attn + io


def wave_bytes(cfg: dict) -> float:
    """Algorithmic HBM bytes of one steady wave: bf16 block weights once,
    window KV reads, own KV writes, latent in/out."""
    n_task = cfg["S"] * cfg["n_streams"]
    d, F, B, C, T, W = cfg["d"], cfg["F"], cfg["B"], cfg["C"], cfg["T"], cfg["W"]
    weights = B * (4 * d * d + 2 * d * F) * 2.0 + 2.0 * C * d
    kv = n_task * B * (W * T * d * 2 * 2 + T * d * 2 * 2)
    latent = n_task * T * C * 4 * 2.0
    return weights + kv + latent


def wave_roofline(cfg: dict, ms_wave: float, peaks: dict, peak_src: str) -> dict:
    """Whole-wave roofline: max(FLOPs at the bf16 peak, bytes at the HBM copy
    rate) against the measured wave time, for the burst and the sustained bf16
    peaks (the timed region is a few hundred ms of back-to-back waves)."""
    flops, bytes_ = wave_flops(cfg), wave_bytes(cfg)
    hbm = peak_value(peaks, "hbm_gbs") * 1e9
    out = {"flops_per_wave": flops, "bytes_per_wave": bytes_,
           "tensor_tflops": flops / (ms_wave / 1e3) / 1e12, "peak_source": peak_src}
    for tag, key in (("burst", "bf16_tflops"), ("sustained", "bf16_tflops_sustained")):
        pk = peak_value(peaks, key) * 1e12
        roof_ms = max(flops / pk, bytes_ / hbm) * 1e3
        out[f"roofline_ms_{tag}"] = roof_ms
        out[f"frac_{tag}"] = roof_ms / ms_wave
    out["frac"] = out["frac_burst"]
    return out


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            with open(p) as f:
                return json.load(f), "measured"
        except Exception:
            pass
    return dict(FALLBACK_PEAKS), "fallback"


def peak_value(peaks: dict, key: str):
    for k in (key, key.replace("_sustained", "")):
        if k in peaks and isinstance(peaks[k], (int, float)):
            return float(peaks[k])
        for v in peaks.values():
            if isinstance(v, dict) and k in v and isinstance(v[k], (int, float)):
                return float(v[k])
    return FALLBACK_PEAKS[key]


class NvmlClocks:
    """SM clock, power and clock-event reasons read through NVML (the driver's
    libnvidia-ml, by ctypes) every 20 ms in a thread during the timed region:
    even a sub-second region gets many samples.  Read-only: no setting of
    the GPU is changed."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, index: int, period_s: float = 0.02):
        import ctypes
        import threading

        self.ct = ctypes
        self.period = period_s
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        self.h = ctypes.c_void_p()
        # the CUDA device's PCI address names the same GPU in NVML whatever
        # CUDA_VISIBLE_DEVICES says; fall back to the index
        found = False
        try:
            import torch

            pr = torch.cuda.get_device_properties(index)
            bus = f"{pr.pci_domain_id:08x}:{pr.pci_bus_id:02x}:{pr.pci_device_id:02x}.0".encode()
            found = self.lib.nvmlDeviceGetHandleByPciBusId_v2(bus, ctypes.byref(self.h)) == 0
        except Exception:
            found = False
        if not found and self.lib.nvmlDeviceGetHandleByIndex_v2(index, ctypes.byref(self.h)) != 0:
            raise RuntimeError("no NVML handle")
        self.reasons_fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
        mx = ctypes.c_uint()
        self.lib.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx))  # 1 = SM clock
        self.max_mhz = float(mx.value)
        self.samples = []
        self._stop = threading.Event()
        self._thread = threading.Thread(target=self._run, daemon=True)

    def _one(self):
        ct = self.ct
        mhz, mw, rs = ct.c_uint(), ct.c_uint(), ct.c_ulonglong()
        self.lib.nvmlDeviceGetClockInfo(self.h, 1, ct.byref(mhz))
        self.lib.nvmlDeviceGetPowerUsage(self.h, ct.byref(mw))
        self.reasons_fn(self.h, ct.byref(rs))
        self.samples.append((float(mhz.value), mw.value / 1000.0, int(rs.value)))

    def _run(self):
        while not self._stop.is_set():
            self._one()
            self._stop.wait(self.period)

    def start(self):
        self._thread.start()

    def stop(self):
        self._stop.set()
        self._thread.join(timeout=5)
        self._one()
        sm = [x[0] for x in self.samples]
        reasons = sorted({n for x in self.samples for bit, n in self.REASONS.items() if x[2] & bit})
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": self.max_mhz, "reasons": reasons,
                "samples": len(sm), "sm_mhz_min": float(min(sm)),
                "power_w_max": float(max(x[1] for x in self.samples)), "source": "nvml, 20 ms"}


class SmiClocks:
    """Fallback: nvidia-smi clock/throttle sampling (200 ms) during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = os.path.join("/tmp", f"psv_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(mx)),
                "reasons": sorted(reasons), "samples": len(sm), "source": "nvidia-smi, 200 ms"}


def ClockSampler(index: int):
    try:
        return NvmlClocks(index)
    except Exception:
        return SmiClocks(index)


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        backend = "nccl" if args.impl == "psv" else "gloo"
        if backend == "nccl":
            import torch

            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def max_over_ranks(x: float, world: int, device=None) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


# ------------------------------------------------------------------ CPU oracle

class OracleWave:
    """One steady wave of the f32 oracle at a configuration's shapes: every
    task at a full window, its block inputs drawn once (seeded) at the
    workload's sizes.  ``block()`` runs the oracle's transformer block for
    every task of the wave once and returns the seconds it took."""

    def __init__(self, cfg: dict):
        from oracle import model as M

        self.M = M
        self.cfg = cfg
        rng = np.random.default_rng(0)
        d, T, W, S = cfg["d"], cfg["T"], cfg["W"], cfg["S"]
        self.n_task = S * cfg["n_streams"]
        specs = dict(synth.block_specs(cfg))
        self.bw = {k: (rng.standard_normal(s, dtype=np.float32) * 0.02 if k.endswith("_w")
                       else np.zeros(s, np.float32)) for k, s in specs.items()}
        self.tasks = []
        for i in range(self.n_task):
            c = W + (S - 1) - (i % S)
            self.tasks.append(dict(
                h=rng.standard_normal((T, d), dtype=np.float32),
                mod=rng.standard_normal(6 * d, dtype=np.float32) * 0.1,
                pos=M.positions(cfg, c),
                window=[(rng.standard_normal((T, d), dtype=np.float32),
                         rng.standard_normal((T, d), dtype=np.float32)) for _ in range(W)]))
        self.threads = os.cpu_count() or 1

    def block(self) -> float:
        t0 = time.perf_counter()
        for t in self.tasks:
            self.M.block_forward(self.cfg, self.bw, t["mod"], t["h"], t["pos"], t["window"])
        return time.perf_counter() - t0


def oracle_wave_sample(cfg: dict, budget_s: float):
    """Time the f32 oracle on blocks of one steady wave until ``budget_s``
    passed (at least one block).  Returns (seconds per whole wave, blocks
    timed, threads)."""
    ow = OracleWave(cfg)
    el, n = 0.0, 0
    while n < cfg["B"] and (n == 0 or el < budget_s):
        el += ow.block()
        n += 1
    return el / n * cfg["B"], n, ow.threads


def run_reference(args, cfg_name, cfg, world, rank):
    """The reference arm: the f32 oracle on the host cores.  One step is one
    transformer block of a steady wave (all tasks at a full window); the
    line's ms_per_step is the measured time of such a step, and the wave
    (all B blocks) is extrapolated from it for ms_per_chunk and value."""
    if rank != 0:
        return 0
    ow = OracleWave(cfg)
    for _ in range(args.warmup):
        ow.block()
    per_step = [ow.block() for _ in range(args.steps)]
    step_s = float(np.mean(per_step))
    wave_s = step_s * cfg["B"]
    value = cfg["n_streams"] / wave_s
    sample = (f"f32 numpy oracle: each step is one transformer block of a steady "
              f"{ow.n_task}-task wave (all tasks at a full W={cfg['W']} window); "
              f"ms_per_chunk and value extrapolate a step x{cfg['B']} blocks")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "chunks/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": step_s * 1e3, "ms_per_chunk": wave_s * 1e3,
        "step": "one transformer block of a steady wave (measured)",
        "extrapolated": {"blocks_per_step": 1, "blocks_per_wave": cfg["B"],
                         "ms_per_wave": wave_s * 1e3, "timed_s": float(np.sum(per_step))},
        "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": workload_name(cfg_name, cfg), "parallelism": "replicas",
                   "l2": "inputs larger than L2"},
        "cpu_baseline": {"value": value, "unit": "chunks/s", "cores": ow.threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "chunks/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ GPU path

def run_psv(args, cfg_name, cfg, world, rank, local):
    import torch

    from autoregressive_denoising_dit_gb300 import Session, _psv as P

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    S, W, T, C = cfg["S"], cfg["W"], cfg["T"], cfg["C"]
    n_st = cfg["n_streams"]
    fill = W + S - 1                       # waves before the first steady wave
    prof_waves = 3
    n_resident = fill + args.warmup + args.steps + prof_waves
    inflight = max(cfg["n_chunks"], n_resident) + S + 8
    sess = Session(cfg, max_streams=n_st, max_inflight=inflight)
    sess.load_device_weights(synth.iter_device_weights(cfg, seed=0, device=f"cuda:{local}"))
    torch.cuda.synchronize()
    streams = synth.make_streams(cfg)
    sids = [sess.open_stream(st.cond) for st in streams]
    # resident inputs: every chunk of the device-timed phase submitted up front
    for c in range(n_resident):
        for st, sid in zip(streams, sids):
            sess.submit(sid, st.noise(c))
    for _ in range(fill + args.warmup):
        sess.run_wave()
    sess.sync(600000)
    torch.cuda.synchronize()

    stream = sess.torch_stream
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    clocks = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize()
    clocks.start()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for k in range(args.steps):
        ev[k][0].record(stream)
        n = sess.run_wave()
        ev[k][1].record(stream)
        assert n == S * n_st, f"wave {k} is not steady ({n} tasks)"
    t1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    barrier(world)
    total_ms = t0.elapsed_time(t1)
    per_wave = sorted(a.elapsed_time(b) for a, b in ev)
    total_ms = max_over_ranks(total_ms, world, dev)
    ms_step = total_ms / args.steps
    value = world * n_st * args.steps / (total_ms / 1e3)

    # per-kernel timing pass (eager launches bracketed by events)
    P.psv_set_profiling(sess.ctx, True)
    for _ in range(prof_waves):
        sess.run_wave()
    times = P.psv_kernel_times(sess.ctx)
    P.psv_set_profiling(sess.ctx, False)
    sess.sync(600000)

    # drain, then the end-to-end phase through host buffers
    while sess.run_wave():
        pass
    sess.sync(600000)
    buf = np.empty((T, C), dtype=np.float32)
    for sid in sids:
        while sess.poll(sid, buf) is not None:
            pass
    next_chunk = n_resident
    e2e_warm = S - 1 + 3
    e2e_steps = args.steps

    # The timed steps' inputs are made beforehand and sit in host memory (the
    # synthetic generator is not part of serving); each step still copies its
    # inputs to the device (submit) and reads its outputs back (poll).
    inputs = {}

    def e2e_submit(c):
        for st, sid in zip(streams, sids):
            sess.submit(sid, inputs[(c, sid)] if (c, sid) in inputs else st.noise(c))
        sess.run_wave()

    def e2e_poll():
        out = 0
        for sid in sids:
            while True:
                got = sess.poll(sid, buf)
                if got is not None:
                    out += 1
                    break
        return out

    for _ in range(e2e_warm):  # pipeline fill: the first S-1 waves emit nothing
        for st, sid in zip(streams, sids):
            sess.submit(sid, st.noise(next_chunk))
        next_chunk += 1
        sess.run_wave()
        for sid in sids:
            sess.poll(sid, buf)
    sess.sync(600000)
    # catch up so each timed step emits exactly one chunk per stream
    for sid in sids:
        while sess.poll(sid, buf) is not None:
            pass
    for c in range(next_chunk, next_chunk + e2e_steps):
        for st, sid in zip(streams, sids):
            inputs[(c, sid)] = np.ascontiguousarray(st.noise(c), dtype=np.float32)
    barrier(world)
    torch.cuda.synchronize()
    # As a server runs it: the next wave (its inputs copied in) is enqueued
    # before the previous wave's outputs are read back, so the device does not
    # wait for the host between waves.  Every one of the K steps' input copies,
    # waves and output reads is inside the clock.
    e2e_clocks = ClockSampler(local)
    e2e_clocks.start()
    w0 = time.perf_counter()
    emitted = 0
    e2e_submit(next_chunk)
    for k in range(1, e2e_steps):
        e2e_submit(next_chunk + k)
        emitted += e2e_poll()
    emitted += e2e_poll()
    next_chunk += e2e_steps
    torch.cuda.synchronize()
    e2e_s_local = time.perf_counter() - w0
    e2e_clk = e2e_clocks.stop()
    assert emitted == n_st * e2e_steps, f"end-to-end phase emitted {emitted} chunks"
    e2e_s = max_over_ranks(e2e_s_local, world, dev)
    e2e_value = world * n_st * e2e_steps / e2e_s
    n_task = S * n_st
    h2d = n_st * T * C * 4 + n_task * 48 + n_st * (cfg["dh"] // 2) * 8
    d2h = n_st * (T * C * 4 + 4)

    # roofline of the dominant kernel
    peaks, peak_src = load_peaks()
    dom = max(times.items(), key=lambda kv: kv[1]["total_ms"])
    name, t = dom
    per_launch_ms = t["total_ms"] / max(1, t["launches"])
    tensor_kernel = name.startswith("gemm") or name == "attention"
    if tensor_kernel:
        achieved = t["flops"] / max(1, t["launches"]) / (per_launch_ms / 1e3) / 1e12
        # the kernel is timed per launch (CUDA events around each launch of a
        # short eager pass): the burst peak is its denominator
        peak = peak_value(peaks, "bf16_tflops")
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak,
                "frac_of_sustained": achieved / peak_value(peaks, "bf16_tflops_sustained")}
    else:
        achieved = t["bytes"] / max(1, t["launches"]) / (per_launch_ms / 1e3) / 1e9
        peak = peak_value(peaks, "hbm_gbs")
        roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak}
    roof["kernel"] = name
    roof["peak_source"] = f"{peak_src} ({'burst bf16' if tensor_kernel else 'HBM copy'})"
    roof["ms_per_launch"] = per_launch_ms
    roof["traffic"] = None
    tfile = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if os.path.exists(tfile):
        try:
            with open(tfile) as f:
                tr = json.load(f)
            ent = tr.get("kernels", {}).get(name)
            if ent and tr.get("config") == cfg_name:
                import hashlib

                with open(os.path.join(ROOT, ent["source"]), "rb") as f:
                    sha = hashlib.sha256(f.read()).hexdigest()[:16]
                # counters of an older build of the kernel do not count
                if sha == ent["sha256_16"]:
                    roof["traffic"] = ent["bytes_per_launch"]
        except Exception:
            pass
    wave_roof = wave_roofline(cfg, ms_step, peaks, peak_src)
    kernels = {k: {"launches": v["launches"], "ms_per_launch": v["total_ms"] / max(1, v["launches"]),
                   "share": v["total_ms"] / max(1e-9, sum(x["total_ms"] for x in times.values()))}
               for k, v in times.items() if v["launches"]}

    line = {
        "metric": METRIC, "value": value, "unit": "chunks/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "ms_per_chunk": ms_step, "ms_per_chunk_p50": per_wave[len(per_wave) // 2],
        "ms_per_chunk_p90": per_wave[min(len(per_wave) - 1, int(0.9 * len(per_wave)))],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic (seeded N(0,0.02) bf16 weights, N(0,1) noise/cond)",
        "config": {"workload": workload_name(cfg_name, cfg), "tasks_per_wave": n_task,
                   "rows_per_wave": n_task * T, "parallelism": "replicas" if world > 1 else "1 GPU",
                   "l2": "inputs larger than L2 (bf16 weights + KV rings read every wave)",
                   "graphs": True},
        "wave_roofline": wave_roof,
        "roofline": roof,
        "kernels": kernels,
        "e2e": {"value": e2e_value, "unit": "chunks/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_s / e2e_steps * 1e3,
                # the SM clock under the power cap during this phase (it runs
                # after the device-timed one; a hotter chip clocks lower)
                "clocks": {k: (e2e_clk or {}).get(k) for k in ("sm_mhz", "sm_mhz_min", "reasons", "samples")}},
        "gpu_launches": (4 + 7 * cfg["B"]) * args.steps,
        "clocks": clk,
        # a chunk's S steps run in S consecutive steady waves
        "response_ms": S * ms_step,
    }
    sess.close()
    del sess
    torch.cuda.empty_cache()
    if world == 1 and not args.no_sweep:
        # every configuration's steady waves (the headline is the one above)
        sweep = {}
        for name in SWEEP:
            if name == cfg_name:
                sweep[name] = {"workload": workload_name(cfg_name, cfg), "steps": args.steps,
                               "ms_per_chunk": ms_step, "chunks_per_s": n_st / (ms_step / 1e3),
                               "wave_frac_burst": wave_roof["frac_burst"],
                               "wave_frac_sustained": wave_roof["frac_sustained"],
                               "tensor_tflops": wave_roof["tensor_tflops"], "headline": True}
                continue
            sweep[name] = measure_steady(name, local)
        line["configs"] = sweep
    if rank == 0 and not args.no_cpu_baseline:
        wave_s, nb, threads = oracle_wave_sample(cfg, args.ref_budget)
        line["cpu_baseline"] = {
            "value": cfg["n_streams"] / wave_s, "unit": "chunks/s", "cores": threads,
            "kind": "oracle",
            "sample": (f"f32 numpy oracle on {nb} transformer block(s) of one steady "
                       f"{n_task}-task wave, scaled x{cfg['B'] / nb:.1f} to the whole wave")}
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def measure_steady(cfg_name: str, local: int, min_seconds: float = 1.5, max_steps: int = 2000,
                   warmup: int = 3) -> dict:
    """ms/chunk of one configuration's steady waves (CUDA graphs, every task at
    a full window), timed with CUDA events over at least ``min_seconds``; the
    attention's time per launch from one eager profiled wave."""
    import torch

    from autoregressive_denoising_dit_gb300 import Session, _psv as P

    cfg = synth.config(cfg_name)
    S, W = cfg["S"], cfg["W"]
    n_st = cfg["n_streams"]
    fill = W + S - 1
    peaks, peak_src = load_peaks()
    est_ms = max(0.05, wave_flops(cfg) / (1.0e15) * 1e3)   # a first guess at 1 PFLOP/s
    steps = int(min(max_steps, max(5, np.ceil(min_seconds * 1e3 / est_ms))))
    n_resident = fill + warmup + 2 * steps + 2
    sess = Session(cfg, max_streams=n_st, max_inflight=n_resident + S + 8)
    try:
        sess.load_device_weights(synth.iter_device_weights(cfg, seed=0, device=f"cuda:{local}"))
        torch.cuda.synchronize()
        streams = synth.make_streams(cfg)
        sids = [sess.open_stream(st.cond) for st in streams]
        rng = np.random.default_rng(7)
        for c in range(n_resident):
            for sid in sids:
                sess.submit(sid, rng.standard_normal((cfg["T"], cfg["C"]), dtype=np.float32))
        for _ in range(fill + warmup):
            sess.run_wave()
        sess.sync(600000)
        stream = sess.torch_stream
        # one timed probe wave sets the step count for the time target
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        sess.run_wave()
        b.record(stream)
        torch.cuda.synchronize()
        steps = int(min(max_steps, max(5, np.ceil(min_seconds / max(1e-6, a.elapsed_time(b) / 1e3)))))
        steps = min(steps, n_resident - fill - warmup - 2)
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for _ in range(steps):
            n = sess.run_wave()
            assert n == S * n_st, f"{cfg_name}: wave is not steady ({n} tasks)"
        t1.record(stream)
        torch.cuda.synchronize()
        ms = t0.elapsed_time(t1) / steps
        P.psv_set_profiling(sess.ctx, True)
        sess.run_wave()
        times = P.psv_kernel_times(sess.ctx)
        P.psv_set_profiling(sess.ctx, False)
        sess.sync(600000)
    finally:
        sess.close()
        torch.cuda.empty_cache()
    at = times.get("attention", {})
    att_us = at.get("total_ms", 0.0) / max(1, at.get("launches", 0)) * 1e3 if at else None
    att_tf = (at["flops"] / at["launches"] / (att_us / 1e6) / 1e12) if at and att_us else None
    roof = wave_roofline(cfg, ms, peaks, peak_src)
    tot = sum(v["total_ms"] for v in times.values()) or 1e-9
    return {"workload": workload_name(cfg_name, cfg), "steps": steps, "ms_per_chunk": ms,
            "chunks_per_s": n_st / (ms / 1e3), "wave_frac_burst": roof["frac_burst"],
            "wave_frac_sustained": roof["frac_sustained"], "tensor_tflops": roof["tensor_tflops"],
            "attention_us_per_launch": att_us, "attention_tflops": att_tf,
            "kernel_us_per_launch": {k: v["total_ms"] / max(1, v["launches"]) * 1e3
                                     for k, v in times.items() if v["launches"]},
            "kernel_share": {k: v["total_ms"] / tot for k, v in times.items() if v["launches"]}}


def run_latency(args, cfg_name, cfg, world, rank, local):
    """Latency-mode schedule (PSV_FLAG_LATENCY): a wave runs each stream's
    oldest ready chunk only, so a chunk's S steps run in S consecutive waves
    of one task per stream.  Reports chunks/s over all streams, the response
    time (first step to output: S such waves, device-timed) and the same
    end to end through host buffers (submit a chunk, run its S waves, poll
    it)."""
    import torch

    from autoregressive_denoising_dit_gb300 import Session, _psv as P

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    S, T, C = cfg["S"], cfg["T"], cfg["C"]
    n_st = cfg["n_streams"]
    n_chunks = args.warmup + args.steps
    sess = Session(cfg, max_streams=n_st, max_inflight=n_chunks + args.steps + S + 8,
                   flags=P.PSV_FLAG_LATENCY)
    sess.load_device_weights(synth.iter_device_weights(cfg, seed=0, device=f"cuda:{local}"))
    torch.cuda.synchronize()
    streams = synth.make_streams(cfg)
    sids = [sess.open_stream(st.cond) for st in streams]
    for c in range(n_chunks):
        for st, sid in zip(streams, sids):
            sess.submit(sid, st.noise(c))
    for _ in range(S * args.warmup):
        sess.run_wave()
    sess.sync(600000)
    stream = sess.torch_stream
    clocks = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize()
    clocks.start()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(S * args.steps):
        n = sess.run_wave()
        assert n == n_st, f"latency-mode wave ran {n} tasks"
    t1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    total_ms = max_over_ranks(t0.elapsed_time(t1), world, dev)
    ms_chunk = total_ms / args.steps          # per stream: one chunk every S waves
    buf = np.empty((T, C), dtype=np.float32)
    for sid in sids:
        while sess.poll(sid, buf) is not None:
            pass
    # end to end: submit one chunk per stream, run its S waves, poll it
    next_chunk = n_chunks
    e2e = []
    for k in range(args.steps + 2):
        # the chunk's input is made before its clock starts (as in the wave e2e)
        noise = [np.ascontiguousarray(st.noise(next_chunk), dtype=np.float32) for st in streams]
        w0 = time.perf_counter()
        for x, sid in zip(noise, sids):
            sess.submit(sid, x)
        for _ in range(S):
            sess.run_wave()
        for sid in sids:
            while sess.poll(sid, buf) is None:
                pass
        if k >= 2:
            e2e.append((time.perf_counter() - w0) * 1e3)
        next_chunk += 1
    e2e_ms = max_over_ranks(float(np.mean(e2e)), world, dev)
    line = {
        "metric": METRIC + " (latency-mode schedule)", "value": world * n_st / (ms_chunk / 1e3),
        "unit": "chunks/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms_chunk, "ms_per_chunk": ms_chunk, "response_ms": ms_chunk,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,0.02) bf16 weights, N(0,1) noise/cond)",
        "config": {"workload": workload_name(cfg_name, cfg), "schedule": "latency (oldest chunk per stream)",
                   "tasks_per_wave": n_st, "rows_per_wave": n_st * T,
                   "parallelism": "replicas" if world > 1 else "1 GPU", "graphs": True},
        "e2e": {"value": world * n_st / (e2e_ms / 1e3), "unit": "chunks/s",
                "h2d_bytes_per_step": n_st * T * C * 4, "d2h_bytes_per_step": n_st * T * C * 4,
                "response_ms": e2e_ms},
        "gpu_launches": (4 + 7 * cfg["B"]) * S * args.steps,
        "clocks": clk,
    }
    sess.close()
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["psv", "reference"], default="psv")
    ap.add_argument("--config", default="wan21_1p3b", choices=sorted(synth.CONFIGS))
    ap.add_argument("--ref-budget", type=float, default=15.0,
                    help="seconds of CPU time for the oracle baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sweep", action="store_true",
                    help="skip the steady-wave timing of the other model configurations")
    ap.add_argument("--latency-mode", action="store_true",
                    help="time the latency-mode schedule (each stream's oldest chunk per wave)")
    ap.add_argument("--blocks", type=int, default=None,
                    help="override the block count (profiling aid: per-block shapes are unchanged)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    cfg = synth.config(args.config)
    if args.blocks:
        cfg["B"] = args.blocks
    world, rank, local = dist_setup(args)
    try:
        if args.impl == "reference":
            return run_reference(args, args.config, cfg, world, rank)
        if args.latency_mode:
            return run_latency(args, args.config, cfg, world, rank, local)
        return run_psv(args, args.config, cfg, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist

            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
