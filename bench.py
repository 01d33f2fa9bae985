#!/usr/bin/env python
"""Throughput of the attention hot path on one GB300 (per rank), one JSON line.

One step = the whole hot path over one batch of synthetic input:
  * causal prefill of the Llama-3.1-8B-shaped workload (B=1, Hq=32, Hkv=8,
    S=2048, d=128, bf16) -- one kernel launch;
  * paged split-KV decode of 64 sequences (lengths U[512, 8192], GQA 32:8,
    d=128, 16-token shuffled pages) -- the split kernel and the combine kernel.
L2 is flushed (a 256 MiB write, then a 256 MiB read) before every step; each launch is bracketed by
CUDA events on the stream it runs on.

Headline value: prefill TFLOP/s (4*B*Hq*d*S(S+1)/2 causal flops / kernel
time); the decode GB/s rides along in "decode".  `e2e` repeats the prefill
metric through the public API with pinned host buffers, host->device copies
of q/k/v and device->host copies of o/lse inside the timed region.

`--impl reference` times the float64 CPU oracle instead (the reference arm:
there is no reference implementation, only the pages' formulas), on a bounded
sample of the same workload, on the host cores.

Multi-GPU: ranks run independent replicas of the workload (no collective on
the data path); value = total work of all ranks / max time over ranks.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import shutil
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from workloads import (LLAMA8B, PAGED, decode_inputs_for, decode_lens_for, decode_min_bytes, make_chunked_inputs,  # noqa
                       make_prefill_inputs, make_varlen_inputs, prefill_inputs_for)

METRIC = "prefill TFLOP/s & decode KV GB/s on 1 GB300, as % of bf16 TC peak / HBM peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
DECODE_SPLITS = 4
E2E_CHUNKS = 4  # query chunks of the pipelined end-to-end prefill
# "GPU Datapath: Where Every Byte Moves in One LLM Inference Step", section C: FA3 on H100 runs this
# exact prefill cell (causal, GQA 32:8, S=2048, d=128) in 87.7 us -> 34.38 GFLOP / 87.7 us.
PAGES_H100_TFLOPS = 34.376515584e9 / 87.7e-6 / 1e12
L2_FLUSH_BYTES = 256 << 20


class L2Flush:
    """A cold, clean L2 before a timed launch: write a buffer larger than L2 (129 MB), which evicts
    every cached line, then read another one, so that the written lines are written back here,
    outside the timed region, and not by the timed kernel.  With the write alone the paged decode
    measured 197.6 us instead of 186.3 us."""

    def __init__(self, dev):
        self.w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
        self.r = torch.ones(L2_FLUSH_BYTES // 8, dtype=torch.int64, device=dev)
        self.sink = torch.empty(1, dtype=torch.int64, device=dev)

    def __call__(self):
        self.w.zero_()
        self.sink.copy_(self.r.sum(dim=0, keepdim=True))


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained")}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def shard(n_units: int, rank: int, world: int) -> range:
    """Contiguous share of n_units for this rank (used when a workload is split over ranks)."""
    base, extra = divmod(n_units, world)
    start = rank * base + min(rank, extra)
    return range(start, start + base + (1 if rank < extra else 0))


class ClockSampler:
    """SM clock and throttle reasons sampled every few ms while the timed region runs.

    Reads NVML through ctypes (no Python package needed); falls back to a
    `nvidia-smi -lms` loop if NVML cannot be loaded.  Reading clocks changes
    nothing on the GPU.
    """

    REASONS = {0x8: "hw_slowdown", 0x40: "hw_thermal_slowdown", 0x20: "sw_thermal_slowdown",
               0x4: "sw_power_cap"}

    def __init__(self, index: int, period_s: float = 0.002):
        self.index = index
        self.period = period_s
        self.samples = []          # (sm_mhz, reasons_mask)
        self.max_mhz = None
        self._stop = threading.Event()
        self._nvml = None
        self._proc = None

    def _open_nvml(self):
        import ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        h = ctypes.c_void_p()
        if lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.index), ctypes.byref(h)) != 0:
            raise OSError("no NVML handle")
        mx = ctypes.c_uint()
        if lib.nvmlDeviceGetMaxClockInfo(h, ctypes.c_int(1), ctypes.byref(mx)) == 0:
            self.max_mhz = float(mx.value)
        self._nvml = (lib, h, ctypes)

    def _loop(self):
        lib, h, ct = self._nvml
        clk, rs = ct.c_uint(), ct.c_ulonglong()
        get_reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
        while not self._stop.is_set():
            if lib.nvmlDeviceGetClockInfo(h, ct.c_int(1), ct.byref(clk)) == 0:
                r = rs.value if get_reasons(h, ct.byref(rs)) == 0 else 0
                self.samples.append((float(clk.value), int(r)))
            time.sleep(self.period)

    def __enter__(self):
        try:
            self._open_nvml()
            self._thread = threading.Thread(target=self._loop, daemon=True)
            self._thread.start()
        except Exception:
            exe = shutil.which("nvidia-smi")
            if exe:
                self._proc = subprocess.Popen(
                    [exe, "-i", str(self.index), "--query-gpu=clocks.sm,clocks.max.sm,clocks_event_reasons.active",
                     "--format=csv,noheader,nounits", "-lms", "20"], stdout=subprocess.PIPE,
                    stderr=subprocess.DEVNULL, text=True)
                self._thread = threading.Thread(target=self._read_smi, daemon=True)
                self._thread.start()
        time.sleep(0.01)
        return self

    def _read_smi(self):
        for line in self._proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            try:
                self.max_mhz = float(parts[1])
                self.samples.append((float(parts[0]), int(parts[2], 16)))
            except (ValueError, IndexError):
                continue

    def __exit__(self, *exc):
        self._stop.set()
        if self._proc:
            self._proc.terminate()
            try:
                self._proc.wait(timeout=5)
            except Exception:
                self._proc.kill()
        if hasattr(self, "_thread"):
            self._thread.join(timeout=2)

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": ["unsampled"]}
        reasons = sorted({name for _, r in self.samples for bit, name in self.REASONS.items() if r & bit})
        return {"sm_mhz": statistics.median(c for c, _ in self.samples), "sm_max_mhz": self.max_mhz,
                "reasons": reasons, "samples": len(self.samples)}


def decode_ws_bytes(attn, max_blocks, cfg, num_splits=0, split_tokens=0):
    """Workspace for one paged decode call (num_splits = split_tokens = 0 is balanced mode)."""
    if num_splits == 0 and split_tokens == 0:
        return attn.decode_balanced_workspace_bytes(cfg.N, cfg.Hq, cfg.Hkv, cfg.d)
    slots = attn.decode_num_slots(max_blocks, num_splits=num_splits, split_tokens=split_tokens)
    return attn.decode_workspace_bytes(cfg.N, cfg.Hq, cfg.d, slots)


def traffic_record(kernel: str):
    """DRAM bytes per launch from a committed ncu summary, if it matches the current kernel source."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f).get(kernel)
    except Exception:
        return None
    if not rec:
        return None
    from attention_attn_prefill_gb300.build import CSRC
    import hashlib
    h = hashlib.sha256()
    for name in rec.get("sources", []):
        with open(os.path.join(CSRC, name), "rb") as f:
            h.update(f.read())
    return rec["bytes_per_launch"] if h.hexdigest() == rec.get("sha256") else None


def run_gpu(args):
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    from attention_attn_prefill_gb300.build import build
    build()
    import attention_attn_prefill_gb300 as attn

    peaks, peak_src = load_peaks()
    cfg = LLAMA8B
    x = prefill_inputs_for(cfg)
    q, k, v = (t.to(dev) for t in (x.q, x.k, x.v))
    o = torch.empty_like(q)
    lse = torch.empty((cfg.B, cfg.Hq, cfg.S), dtype=torch.float32, device=dev)

    dcfg = PAGED
    lens = decode_lens_for(dcfg)
    dx = decode_inputs_for(dcfg)
    dq, kc, vc, bt, sl = (t.to(dev) for t in (dx.q, dx.k_cache, dx.v_cache, dx.block_table, dx.seq_lens))
    do = torch.empty_like(dq)
    dl = torch.empty((dcfg.N, dcfg.Hq), dtype=torch.float32, device=dev)
    ws = torch.empty(max(1, decode_ws_bytes(attn, dx.max_blocks, dcfg, num_splits=args.decode_splits)),
                     dtype=torch.uint8, device=dev)
    slots = attn.decode_num_slots(dx.max_blocks, num_splits=args.decode_splits) if args.decode_splits else 0
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream(dev)

    def prefill():
        attn.prefill(q, k, v, scale=cfg.scale, causal=True, out=o, lse=lse, stream=stream)

    def decode():
        attn.decode_paged(dq, kc, vc, bt, sl, scale=dcfg.scale, num_splits=args.decode_splits, out=do, lse=dl,
                          workspace=ws, stream=stream)

    def step(record):
        flush()
        e0, e1, e2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
        e0.record(stream)
        prefill()
        e1.record(stream)
        decode()
        e2.record(stream)
        record.append((e0, e1, e2))

    warm = []
    for _ in range(args.warmup):
        step(warm)
    torch.cuda.synchronize()
    assert attn.device_status(clear=True) == 0
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    rec = []
    with ClockSampler(local) as clocks:
        t0 = time.perf_counter()
        for _ in range(args.steps):
            step(rec)
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
    if world > 1:
        torch.distributed.barrier()
    pre_ms = [a.elapsed_time(b) for a, b, _ in rec]
    dec_ms = [b.elapsed_time(c) for _, b, c in rec]
    spread = {"prefill_us": {"mean": round(statistics.mean(pre_ms) * 1e3, 2),
                             "median": round(statistics.median(pre_ms) * 1e3, 2), "min": round(min(pre_ms) * 1e3, 2)},
              "decode_us": {"mean": round(statistics.mean(dec_ms) * 1e3, 2),
                            "median": round(statistics.median(dec_ms) * 1e3, 2), "min": round(min(dec_ms) * 1e3, 2)}}
    pre_mean, dec_mean = statistics.mean(pre_ms), statistics.mean(dec_ms)
    step_ms = pre_mean + dec_mean
    if world > 1:
        t = torch.tensor([pre_mean, dec_mean, step_ms], device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        pre_mean, dec_mean, step_ms = t.tolist()

    flops = cfg.causal_flops
    tflops = world * flops / (pre_mean * 1e-3) / 1e12
    dbytes = decode_min_bytes(lens, dcfg.Hq, dcfg.Hkv, dcfg.d)
    gbs = world * dbytes / (dec_mean * 1e-3) / 1e9

    # ---- end to end through the public API with host buffers (prefill metric)
    hq, hk, hv = (t.pin_memory() for t in (x.q, x.k, x.v))
    ho = torch.empty(o.shape, dtype=o.dtype, pin_memory=True)
    hl = torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True)
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv))
    d2h = ho.numel() * ho.element_size() + hl.numel() * hl.element_size()

    def e2e_serial():
        q.copy_(hq, non_blocking=True)
        k.copy_(hk, non_blocking=True)
        v.copy_(hv, non_blocking=True)
        prefill()
        ho.copy_(o, non_blocking=True)
        hl.copy_(lse, non_blocking=True)

    # the library's host-buffer prefill: the transfers overlap the chunks' compute inside the call
    hq1, hk1, hv1, ho1 = (t[0] for t in (hq, hk, hv, ho))   # one sequence, [S, H, d]
    hl1 = hl[0]
    ws_host = torch.empty(attn.prefill_host_workspace_bytes(cfg.S, cfg.Hq, cfg.Hkv, cfg.d, E2E_CHUNKS),
                          dtype=torch.uint8, device=dev)

    def e2e_host():
        attn.prefill_host(hq1, hk1, hv1, scale=cfg.scale, causal=True, chunks=E2E_CHUNKS, out=ho1, lse=hl1,
                          workspace=ws_host, stream=stream)

    def timed_e2e(step_fn):
        for _ in range(args.warmup):
            step_fn()
        torch.cuda.synchronize()
        ev = []
        for _ in range(args.steps):
            flush()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            step_fn()
            b.record(stream)
            ev.append((a, b))
        torch.cuda.synchronize()
        return statistics.mean(a.elapsed_time(b) for a, b in ev)

    e2e_ms = timed_e2e(e2e_host)
    e2e_serial_ms = timed_e2e(e2e_serial)
    if world > 1:
        t = torch.tensor([e2e_ms], device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        e2e_ms = t.item()
    e2e_tflops = world * flops / (e2e_ms * 1e-3) / 1e12
    status = attn.device_status(clear=True)

    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return
    achieved = flops / (statistics.mean(pre_ms) * 1e-3) / 1e12
    peak_tc = peaks["bf16_tflops"]
    dec_achieved = dbytes / (statistics.mean(dec_ms) * 1e-3) / 1e9
    launches_per_step = 1 + 1 + (1 if (slots > 1 or args.decode_splits == 0) else 0)
    dec_roof = {"bound": "hbm", "kernel": "decode_split_kernel<128,4,2> + combine_kernel<128>",
                "achieved": round(dec_achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(dec_achieved / peaks["hbm_gbs"], 4), "frac_of_8tbs": round(dec_achieved / 8000.0, 4),
                "peak_source": f"{peak_src} HBM copy", "traffic": traffic_record("decode_split_kernel<128,4,2>"),
                "share_of_step": round(dec_mean / step_ms, 3),
                "note": "one decode call: split kernel + combine, timed together"}
    line = {
        "metric": METRIC,
        "value": round(tflops, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(step_ms, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": round(tflops / PAGES_H100_TFLOPS, 3),
        "vs_baseline_ref": f"{PAGES_H100_TFLOPS:.1f} TFLOP/s: FA3 on H100, 87.7 us for this prefill cell (pages)",
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16; shapes of the pages' workloads)",
        "config": {
            "workload": "causal prefill B=1 Hq=32 Hkv=8 S=2048 d=128 + paged decode N=64 len~U[512,8192] "
                        f"Hq=32 Hkv=8 d=128 num_splits={args.decode_splits}",
            "prefill": {"B": cfg.B, "Hq": cfg.Hq, "Hkv": cfg.Hkv, "S": cfg.S, "d": cfg.d, "causal": True,
                        "seed": cfg.seed, "flops_per_step": flops},
            "decode": {"N": dcfg.N, "Hq": dcfg.Hq, "Hkv": dcfg.Hkv, "d": dcfg.d, "page": 16,
                       "num_splits": args.decode_splits, "slots": slots, "sum_len": int(sum(lens)),
                       "seed": dcfg.seed, "bytes_per_step": dbytes},
            "l2": "flushed between steps: a 256 MiB write, then a 256 MiB read, outside the timed events",
            "parallelism": f"replicas x{world}",
        },
        # the dominant kernel of the step by time is the decode (split + combine: about 85% of the
        # step); its roofline leads, the prefill's follows under "prefill"
        "roofline": dec_roof,
        "prefill": {
            "value": round(tflops, 2), "unit": "TFLOP/s", "ms": round(pre_mean, 4),
            "roofline": {
                "bound": "tensor", "kernel": "prefill_cta2_kernel", "achieved": round(achieved, 2),
                "peak": peak_tc, "unit": "TFLOP/s", "frac": round(achieved / peak_tc, 4),
                "peak_source": f"{peak_src} bf16 dense (burst)",
                "traffic": traffic_record("prefill_cta2_kernel"), "algorithmic_bytes": cfg.min_bytes,
            },
            "flops_convention": "exact causal pairs, 4*B*Hq*d*S(S+1)/2",
            "s2_over_2": {"flops_per_step": cfg.s2_flops,
                          "TFLOP/s": round(world * cfg.s2_flops / (pre_mean * 1e-3) / 1e12, 2)},
        },
        "timing_spread": spread,
        "decode": {"value": round(gbs, 1), "unit": "GB/s", "ms": round(dec_mean, 4), "roofline": dec_roof},
        "e2e": {"value": round(e2e_tflops, 2), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms": round(e2e_ms, 4),
                "how": f"one attn_prefill_host call a step: q/k/v read from pinned host memory and o/lse "
                       f"written back to it inside the call, pipelined in {E2E_CHUNKS} query chunks (each a "
                       "chunked prefill over the sequence's own keys) with the copies on two library "
                       "streams",
                "serial": {"value": round(world * flops / (e2e_serial_ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
                           "ms": round(e2e_serial_ms, 4), "how": "copies in, one attn_prefill, copies out, "
                                                                 "in sequence on one stream",
                           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks.summary(),
        "wall_s_timed": round(wall, 3),
        "device_status": status,
    }
    if not args.no_workloads:
        line["workloads"] = workload_table(attn, dev, stream, flush, peaks, (dx, (dq, kc, vc, bt, sl)))
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def workload_table(attn, dev, stream, flush, peaks, paged_inputs, reps: int = 50):
    """Every seeded workload (outside the timed region): `reps` launches, L2 flushed before each.

    Each entry's value is from the mean launch time; the median and the fastest launch ride along."""
    from workloads import DECODE_CONFIGS, PREFILL_CONFIGS
    spread = {}

    def timed(launch):
        launch()
        torch.cuda.synchronize()
        ms = []
        for _ in range(reps):
            flush()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            launch()
            b.record(stream)
            ms.append((a, b))
        torch.cuda.synchronize()
        t = [a.elapsed_time(b) for a, b in ms]
        spread["us_median"] = round(statistics.median(t) * 1e3, 1)
        spread["us_min"] = round(min(t) * 1e3, 1)
        return statistics.mean(t)

    out = {}
    for cfg in PREFILL_CONFIGS:
        x = prefill_inputs_for(cfg)
        q, k, v = (t.to(dev) for t in (x.q, x.k, x.v))
        o = torch.empty_like(q)
        lse = torch.empty((cfg.B, cfg.Hq, cfg.S), dtype=torch.float32, device=dev)
        ms = timed(lambda: attn.prefill(q, k, v, scale=cfg.scale, causal=True, out=o, lse=lse, stream=stream))
        tf = cfg.causal_flops / (ms * 1e-3) / 1e12
        out[cfg.name] = {"TFLOP/s": round(tf, 1), "us": round(ms * 1e3, 1), **spread,
                         "frac": round(tf / peaks["bf16_tflops"], 4),
                         "TFLOP/s_s2_over_2": round(cfg.s2_flops / (ms * 1e-3) / 1e12, 1)}
        del q, k, v, o, lse
    for cfg in DECODE_CONFIGS:
        if cfg.name == "paged_decode":
            x, (dq, kc, vc, bt, sl) = paged_inputs
        else:
            x = decode_inputs_for(cfg)
            dq, kc, vc, bt, sl = (t.to(dev) for t in (x.q, x.k_cache, x.v_cache, x.block_table, x.seq_lens))
        lens = decode_lens_for(cfg)
        nbytes = decode_min_bytes(lens, cfg.Hq, cfg.Hkv, cfg.d)
        do = torch.empty_like(dq)
        dl = torch.empty((cfg.N, cfg.Hq), dtype=torch.float32, device=dev)
        specs = [dict(num_splits=n) for n in cfg.num_splits] + [dict(split_tokens=t) for t in cfg.split_tokens]
        auto_t = attn.decode_auto_split_tokens(lens, cfg.Hkv, cfg.d, x.max_blocks)
        specs += [dict(split_tokens=auto_t),
                  dict(num_splits=attn.decode_auto_splits(cfg.N, cfg.Hkv, cfg.d, x.max_blocks)),
                  dict(num_splits=0)]
        names = [f"splits={sp['num_splits']}" if "num_splits" in sp else f"split_tokens={sp['split_tokens']}"
                 for sp in specs]
        names[-3] = f"auto (length-aware, {auto_t}-token groups)"
        names[-2] = f"FA2 rule ({specs[-2]['num_splits']} splits)"
        names[-1] = "balanced"
        for name, sp in zip(names, specs):
            ws = torch.empty(max(1, decode_ws_bytes(attn, x.max_blocks, cfg, **sp)), dtype=torch.uint8, device=dev)
            ms = timed(lambda: attn.decode_paged(dq, kc, vc, bt, sl, scale=cfg.scale, out=do, lse=dl, workspace=ws,
                                                 stream=stream, **sp))
            gbs = nbytes / (ms * 1e-3) / 1e9
            out[f"{cfg.name} {name}"] = {"GB/s": round(gbs, 1), "us": round(ms * 1e3, 1), **spread,
                                         "frac": round(gbs / peaks["hbm_gbs"], 4)}
        # other backends' decode numerics, with the group counts they would pick on this GPU
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        for backend in attn.NUMERICS:
            parts = attn.emulated_partitions(backend, cfg.N, cfg.Hkv, max(lens), sms)
            slots = attn.emulated_num_slots(backend, x.max_blocks, parts)
            ws = torch.empty(attn.lib().attn_emulated_workspace_bytes(cfg.N, cfg.Hq, cfg.d, slots),
                             dtype=torch.uint8, device=dev)
            ms = timed(lambda: attn.decode_paged_emulated(dq, kc, vc, bt, sl, numerics=backend, partitions=parts,
                                                          scale=cfg.scale, out=do, lse=dl, workspace=ws,
                                                          stream=stream))
            gbs = nbytes / (ms * 1e-3) / 1e9
            out[f"{cfg.name} emulated {backend} ({slots} groups)"] = {
                "GB/s": round(gbs, 1), "us": round(ms * 1e3, 1), **spread, "frac": round(gbs / peaks["hbm_gbs"], 4)}
            del ws
    # packed sequences of mixed lengths and chunked prefill over a paged cache, Llama-8B heads
    Hq, Hkv, d = 32, 8, 128
    lens = [int(v) for v in torch.randint(256, 4097, (8,), generator=torch.Generator().manual_seed(12))]
    xv = make_varlen_inputs(lens, Hq=Hq, Hkv=Hkv, d=d, seed=12)
    vq, vk, vv, vcu = (t.to(dev) for t in (xv.q, xv.k, xv.v, xv.cu_seqlens))
    vo = torch.empty_like(vq)
    vl = torch.empty((Hq, vq.shape[0]), dtype=torch.float32, device=dev)
    ms = timed(lambda: attn.prefill_varlen(vq, vk, vv, vcu, xv.max_seqlen, scale=d ** -0.5, out=vo, lse=vl,
                                           stream=stream))
    flops = 4.0 * Hq * d * sum(L * (L + 1) / 2 for L in lens)
    out[f"packed prefill, 8 sequences of {min(lens)}-{max(lens)} tokens"] = {
        "TFLOP/s": round(flops / (ms * 1e-3) / 1e12, 1), "us": round(ms * 1e3, 1), **spread,
        "frac": round(flops / (ms * 1e-3) / 1e12 / peaks["bf16_tflops"], 4)}
    del vq, vk, vv, vo, vl
    for n, qn, ctxn in ((4, 2048, 8192), (16, 512, 4096)):
        xc = make_chunked_inputs([ctxn] * n, [qn] * n, Hq=Hq, Hkv=Hkv, d=d, seed=11)
        cargs = [t.to(dev) for t in (xc.q, xc.k_cache, xc.v_cache, xc.block_table, xc.cu_seqlens_q, xc.seq_lens)]
        co = torch.empty_like(cargs[0])
        cl = torch.empty((Hq, xc.q.shape[0]), dtype=torch.float32, device=dev)
        ms = timed(lambda: attn.prefill_paged(*cargs, xc.max_seqlen_q, scale=d ** -0.5, causal=True, out=co, lse=cl,
                                              stream=stream))
        flops = 4.0 * Hq * d * n * sum(ctxn - qn + i + 1 for i in range(qn))
        out[f"chunked prefill, {n} x {qn} new tokens over {ctxn}-token contexts"] = {
            "TFLOP/s": round(flops / (ms * 1e-3) / 1e12, 1), "us": round(ms * 1e3, 1), **spread,
            "frac": round(flops / (ms * 1e-3) / 1e12 / peaks["bf16_tflops"], 4)}
        del cargs, co, cl
    # a batch whose keys and values (268 MB) exceed L2: MHA, 4 x 32 heads, S = 4096 (blocked walk)
    xm = make_prefill_inputs(4, 32, 32, 4096, 128, seed=13)
    mq, mk, mv = (t.to(dev) for t in (xm.q, xm.k, xm.v))
    mo = torch.empty_like(mq)
    ml = torch.empty((4, 32, 4096), dtype=torch.float32, device=dev)
    ms = timed(lambda: attn.prefill(mq, mk, mv, scale=d ** -0.5, causal=True, out=mo, lse=ml, stream=stream))
    flops = 4.0 * 4 * 32 * d * 4096 * 4097 / 2
    out["MHA prefill, 4 x 32 heads, S = 4096 (K+V 268 MB, larger than L2)"] = {
        "TFLOP/s": round(flops / (ms * 1e-3) / 1e12, 1), "us": round(ms * 1e3, 1), **spread,
        "frac": round(flops / (ms * 1e-3) / 1e12 / peaks["bf16_tflops"], 4)}
    del mq, mk, mv, mo, ml
    out["_note"] = (f"each: {reps} launches with L2 flushed before each, outside the timed region; value and frac "
                    "from the mean launch time (us), with the median and the fastest launch beside it; frac against "
                    "the measured bf16 dense peak (prefill) or HBM copy (decode); prefill flops count the causal "
                    "(query, key) pairs exactly, S(S+1)/2 per head, and TFLOP/s_s2_over_2 repeats the value under "
                    "the S^2/2 convention")
    if attn.device_status(clear=True) != 0:
        out["_device_status"] = "nonzero"
    return out


# ---------------------------------------------------------------------------- CPU oracle

def cpu_baseline(min_seconds: float):
    """Oracle on whole query heads of the prefill workload, repeated until about min_seconds of work."""
    import oracle.attention as oa
    cfg = LLAMA8B
    x = prefill_inputs_for(cfg)
    heads, t0 = 0, time.perf_counter()
    while time.perf_counter() - t0 < min_seconds and heads < 4 * cfg.Hq:
        oa.prefill(x.q, x.k, x.v, cfg.scale, causal=True, heads=[heads % cfg.Hq])
        heads += 1
    dt = time.perf_counter() - t0
    flops = cfg.causal_flops * heads / cfg.Hq
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"float64 numpy oracle, causal prefill B=1 S=2048 d=128: {heads} query-head passes "
                      f"(all 2048 rows each) in {dt:.2f} s, {flops / 1e9:.1f} GFLOP counted causally; "
                      "numpy BLAS threads = host cores",
            "single_core_tiny": single_core_tiny()}


def single_core_tiny(seconds: float = 1.0):
    """The oracle on the tiny config (B=1, S=128, d=64) on one host core: a child process with every
    BLAS/OpenMP thread pool set to one thread, repeated for about `seconds`."""
    code = (
        "import time, oracle.attention as oa\n"
        "from workloads import TINY, prefill_inputs_for\n"
        "x = prefill_inputs_for(TINY)\n"
        "oa.prefill(x.q, x.k, x.v, TINY.scale, causal=True)\n"
        "n, t0 = 0, time.perf_counter()\n"
        f"while time.perf_counter() - t0 < {seconds}:\n"
        "    oa.prefill(x.q, x.k, x.v, TINY.scale, causal=True); n += 1\n"
        "dt = time.perf_counter() - t0\n"
        "print(n, dt, TINY.causal_flops)\n")
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               NUMEXPR_NUM_THREADS="1", CUDA_VISIBLE_DEVICES="")
    try:
        out = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True, text=True,
                             timeout=120, check=True).stdout.split()
        n, dt, fl = int(out[0]), float(out[1]), float(out[2])
    except Exception as exc:  # reported, not fatal: the multi-core figure above stands
        return {"error": str(exc)[:200]}
    return {"value": n * fl / dt / 1e12, "unit": "TFLOP/s", "cores": 1,
            "sample": f"tiny causal prefill B=1 Hq=1 S=128 d=64, {n} passes in {dt:.2f} s, one thread",
            "ms_per_pass": round(1e3 * dt / n, 3)}


def run_reference(args):
    """The float64 oracle on the host cores: each step is `ref_heads` query heads of the prefill workload."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle.attention as oa
    cfg = LLAMA8B
    x = prefill_inputs_for(cfg)

    def step(i):
        heads = [(i * args.ref_heads + h) % cfg.Hq for h in range(args.ref_heads)]
        oa.prefill(x.q, x.k, x.v, cfg.scale, causal=True, heads=heads)

    for i in range(args.warmup):
        step(i)
    t_all = time.perf_counter()
    for i in range(args.steps):
        step(i)
    total = time.perf_counter() - t_all
    value = args.steps * LLAMA8B.causal_flops * args.ref_heads / LLAMA8B.Hq / total / 1e12
    line = {
        "metric": METRIC, "impl": "reference", "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) bf16 inputs widened to float64)",
        "config": {"workload": "causal prefill B=1 Hq=32 Hkv=8 S=2048 d=128 (sample of query heads per step)",
                   "heads_per_step": args.ref_heads},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
                         "sample": f"{args.ref_heads} of 32 query heads per step, all 2048 rows"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_case(args):
    """One kernel family on one named workload, for profiling: prints a short JSON line.

    prefill:<name>            name in {tiny, llama8b_prefill, sweep_s1024, sweep_s2048, sweep_s4096,
                              qwen_d256_prefill}
    shape:<B>x<Hq>x<Hkv>x<S>x<d>  causal prefill of that shape (seeded N(0,1) inputs)
    varlen:<mix|L1,L2,..>[:<Hq>x<Hkv>x<d>]  packed sequences: the workload table's mix (8 sequences)
                              or the given lengths (Llama-8B heads unless given)
    chunked:<n>x<q>of<ctx>[:<Hq>x<Hkv>x<d>]  chunked prefill against the paged cache (Llama-8B heads
                              unless given): n sequences of ctx cached tokens whose last q are new
    decode:<name>:<splits>    name in {paged_decode, longctx_decode}; splits = num_splits (0 = balanced
                              mode), t<N> for split_tokens = N, auto for the FA2 split-count rule, or
                              autot for the length-aware group size
    decode_emu:<name>:<backend>  the same workloads with another backend's numerics (triton, fa2, xqa,
                              trt) and the group count it would pick on this GPU
    """
    from workloads import DECODE_CONFIGS, PREFILL_CONFIGS
    from attention_attn_prefill_gb300.build import build
    build()
    import attention_attn_prefill_gb300 as attn
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev)
    kind, name, *rest = args.case.split(":")
    if kind == "shape":
        # a causal prefill of any shape: name = "<B>x<Hq>x<Hkv>x<S>x<d>" (odd Hq / Hkv takes the
        # single-head kernel at d = 128)
        B, Hq, Hkv, S, d = (int(v) for v in name.split("x"))
        x = make_prefill_inputs(B, Hq, Hkv, S, d, seed=21)
        q, k, v = (t.to(dev) for t in (x.q, x.k, x.v))
        o = torch.empty_like(q)
        lse = torch.empty((B, Hq, S), dtype=torch.float32, device=dev)
        work, unit = 4.0 * B * Hq * d * S * (S + 1) / 2 / 1e12, "TFLOP/s"

        def launch():
            attn.prefill(q, k, v, scale=d ** -0.5, causal=True, out=o, lse=lse, stream=stream)
    elif kind == "varlen":
        # name "mix": the packed mix of the workload table (8 sequences of seeded lengths U[256, 4096]);
        # else comma-separated lengths; Llama-8B heads unless <Hq>x<Hkv>x<d> follows
        Hq, Hkv, d = (int(v) for v in rest[0].split("x")) if rest else (32, 8, 128)
        if name == "mix":
            lens = [int(v) for v in torch.randint(256, 4097, (8,), generator=torch.Generator().manual_seed(12))]
        else:
            lens = [int(v) for v in name.split(",")]
        xv = make_varlen_inputs(lens, Hq=Hq, Hkv=Hkv, d=d, seed=12)
        vq, vk, vv, vcu = (t.to(dev) for t in (xv.q, xv.k, xv.v, xv.cu_seqlens))
        vo = torch.empty_like(vq)
        vl = torch.empty((Hq, vq.shape[0]), dtype=torch.float32, device=dev)
        work, unit = 4.0 * Hq * d * sum(L * (L + 1) / 2 for L in lens) / 1e12, "TFLOP/s"

        def launch():
            attn.prefill_varlen(vq, vk, vv, vcu, xv.max_seqlen, scale=d ** -0.5, out=vo, lse=vl, stream=stream)
    elif kind == "chunked":
        # chunked prefill against the paged cache: <n> sequences of <ctx> cached tokens, the last <q> new
        # (name = "<n>x<q>of<ctx>"), Llama-8B heads
        n, rest_ = name.split("x")
        qn, ctxn = (int(v) for v in rest_.split("of"))
        n = int(n)
        Hq, Hkv, d = (int(v) for v in rest[0].split("x")) if rest else (32, 8, 128)
        x = make_chunked_inputs([ctxn] * n, [qn] * n, Hq=Hq, Hkv=Hkv, d=d, seed=11)
        args_ = [t.to(dev) for t in (x.q, x.k_cache, x.v_cache, x.block_table, x.cu_seqlens_q, x.seq_lens)]
        o = torch.empty_like(args_[0])
        lse = torch.empty((Hq, x.q.shape[0]), dtype=torch.float32, device=dev)
        pairs = n * sum(ctxn - qn + i + 1 for i in range(qn))
        work, unit = 4.0 * Hq * d * pairs / 1e12, "TFLOP/s"

        def launch():
            attn.prefill_paged(*args_, x.max_seqlen_q, scale=1.0 / math.sqrt(d), causal=True, out=o, lse=lse,
                               stream=stream)
    elif kind == "prefill":
        cfg = {c.name: c for c in PREFILL_CONFIGS}[name]
        x = prefill_inputs_for(cfg)
        q, k, v = (t.to(dev) for t in (x.q, x.k, x.v))
        o = torch.empty_like(q)
        lse = torch.empty((cfg.B, cfg.Hq, cfg.S), dtype=torch.float32, device=dev)
        work, unit = cfg.causal_flops / 1e12, "TFLOP/s"

        def launch():
            attn.prefill(q, k, v, scale=cfg.scale, causal=True, out=o, lse=lse, stream=stream)
    elif kind == "decode_emu":
        cfg = {c.name: c for c in DECODE_CONFIGS}[name]
        backend = rest[0]
        lens = decode_lens_for(cfg)
        x = decode_inputs_for(cfg)
        dq, kc, vc, bt, sl = (t.to(dev) for t in (x.q, x.k_cache, x.v_cache, x.block_table, x.seq_lens))
        do = torch.empty_like(dq)
        dl = torch.empty((cfg.N, cfg.Hq), dtype=torch.float32, device=dev)
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        parts = attn.emulated_partitions(backend, cfg.N, cfg.Hkv, max(lens), sms)
        slots = attn.emulated_num_slots(backend, x.max_blocks, parts)
        ws = torch.empty(attn.lib().attn_emulated_workspace_bytes(cfg.N, cfg.Hq, cfg.d, slots), dtype=torch.uint8,
                         device=dev)
        work, unit = decode_min_bytes(lens, cfg.Hq, cfg.Hkv, cfg.d) / 1e9, "GB/s"

        def launch():
            attn.decode_paged_emulated(dq, kc, vc, bt, sl, numerics=backend, partitions=parts, scale=cfg.scale,
                                       out=do, lse=dl, workspace=ws, stream=stream)
    else:
        cfg = {c.name: c for c in DECODE_CONFIGS}[name]
        spec = rest[0] if rest else "1"
        lens = decode_lens_for(cfg)
        x = decode_inputs_for(cfg)
        if spec == "auto":
            kw = dict(num_splits=attn.decode_auto_splits(cfg.N, cfg.Hkv, cfg.d, x.max_blocks))
        elif spec == "autot":
            kw = dict(split_tokens=attn.decode_auto_split_tokens(lens, cfg.Hkv, cfg.d, x.max_blocks))
        elif spec.startswith("t"):
            kw = dict(split_tokens=int(spec[1:]))
        else:
            kw = dict(num_splits=int(spec))
        dq, kc, vc, bt, sl = (t.to(dev) for t in (x.q, x.k_cache, x.v_cache, x.block_table, x.seq_lens))
        do = torch.empty_like(dq)
        dl = torch.empty((cfg.N, cfg.Hq), dtype=torch.float32, device=dev)
        ws = torch.empty(max(1, decode_ws_bytes(attn, x.max_blocks, cfg, **kw)), dtype=torch.uint8, device=dev)
        work, unit = decode_min_bytes(lens, cfg.Hq, cfg.Hkv, cfg.d) / 1e9, "GB/s"

        def launch():
            attn.decode_paged(dq, kc, vc, bt, sl, scale=cfg.scale, out=do, lse=dl, workspace=ws, stream=stream,
                              **kw)
    flush = L2Flush(dev)
    for _ in range(args.warmup):
        flush()
        launch()
    torch.cuda.synchronize()
    ms = []
    for _ in range(args.steps):
        flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        launch()
        b.record(stream)
        ms.append((a, b))
    torch.cuda.synchronize()
    t = [a.elapsed_time(b) for a, b in ms]
    status = attn.device_status(clear=True)
    print(json.dumps({"case": args.case, "ms_mean": statistics.mean(t), "ms_min": min(t),
                      "value": work / (statistics.mean(t) * 1e-3), "best": work / (min(t) * 1e-3), "unit": unit,
                      "device_status": status}), flush=True)
    if status:
        sys.exit(3)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("gb300", "reference"), default="gb300")
    ap.add_argument("--decode-splits", type=int, default=DECODE_SPLITS)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--ref-heads", type=int, default=1)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-workloads", action="store_true", help="skip the per-workload table")
    ap.add_argument("--case", default="", help="profile one kernel on one workload (see run_case)")
    args = ap.parse_args()
    if args.case:
        return run_case(args)
    args.warmup = max(3, args.warmup)   # at least three untimed warm-up steps
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
