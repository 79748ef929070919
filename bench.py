#!/usr/bin/env python3
"""Benchmark of the CacheGen codec's hot path on GB300.

One step = encode + decode of one synthetic KV blob that is already in HBM
(quantise, histograms/CDFs, arithmetic coding, packing; then prefix-sum
decoding with fused dequantisation). The metric is GB/s of raw bf16 KV per
step; encode and decode GB/s, the compression ratio, the dominant kernel's
HBM roofline fraction, an end-to-end figure through host buffers, and the
CPU oracle's speed on the host cores are reported beside it.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...   # the CPU oracle as the reference arm

Under torchrun (N > 1) every rank encodes and decodes its own replica of
the workload (weak scaling; the codec has no exchange step), the ranks
barrier around the timed region, and rank 0 reports the slowest rank's
time.
"""
from __future__ import annotations

import argparse
import hashlib
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
# The CPU baseline's OpenMP threads sleep once their work is done instead of
# spinning, so they take no host cycles from the end-to-end leg that follows.
os.environ.setdefault("OMP_WAIT_POLICY", "PASSIVE")

METRIC = "CacheGen encode+decode throughput (GB/s of raw bf16 KV)"
DEFAULT_WORKLOAD = "llama8b_t16k"
KERNEL_SOURCE = os.path.join(ROOT, "kv_cache_compression_03_gb300", "csrc", "cachegen_kernels.cu")


# ----------------------------------------------------------------- ranks

def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def aggregate_max(value: float, world: int, backend_device=None) -> float:
    """Max of a float over all ranks (identity for one rank)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=backend_device or "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while it runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 20):
        self.gpu = gpu_index
        self.period = period_ms
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", f"-lms={self.period}"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
            # let sampling start before the timed region (a short region may
            # otherwise end before nvidia-smi prints its first line)
            t_end = time.perf_counter() + 3.0
            while not self.lines and self.proc.poll() is None and time.perf_counter() < t_end:
                time.sleep(0.005)
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
            self._t.join(timeout=2)

    def summary(self):
        if not self.lines:
            return None
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower() in ("active", "1", "yes"):
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------- workload

def workload_info(name: str):
    from kv_cache_compression_03_gb300 import synthetic
    p = synthetic.WORKLOADS[name]
    k, v = synthetic.workload_specs(name)
    return p, k, v


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def code_hash(text: str) -> str:
    """sha256 of C/CUDA source with comments and whitespace removed, so that
    an edit of comments alone keeps the hash (string literals in the kernel
    source hold no comment markers)."""
    import re
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    text = re.sub(r"\s+", "", text)
    return hashlib.sha256(text.encode()).hexdigest()[:16]


def kernel_source_hash() -> str:
    with open(KERNEL_SOURCE, encoding="utf-8") as f:
        return code_hash(f.read())


def recorded_counter(kernel: str, workload: str, key: str = "dram_bytes_per_launch"):
    """A per-launch counter (DRAM bytes, warp instructions) from a committed
    ncu capture, if it was taken on the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    e = d.get(kernel, {}).get(workload)
    if not e or e.get("source_sha") != kernel_source_hash():
        return None
    return e.get(key)


NOMINAL_SM_MHZ = 2070.0  # maximum SM clock of the part when nvidia-smi is unavailable


def issue_ceiling(kernel: str, workload: str, ms_per_launch: float, sms: int, sm_mhz):
    """The coders are bound by instruction issue, not HBM: warp instructions
    per launch (ncu, current source) over the launch time, against one warp
    instruction per scheduler per cycle (4 per SM) at the maximum SM clock."""
    inst = recorded_counter(kernel, workload, "warp_instructions_per_launch")
    mhz = float(sm_mhz) if sm_mhz else NOMINAL_SM_MHZ
    peak = sms * 4 * mhz * 1e6
    if inst is None:
        return {"bound": "alu", "kernel": kernel, "achieved": None, "peak": peak,
                "unit": "warp-instructions/s", "frac": None, "instructions_per_launch": None}
    achieved = inst / (ms_per_launch * 1e-3)
    return {"bound": "alu", "kernel": kernel, "achieved": round(achieved / 1e9, 2) * 1e9,
            "peak": peak, "unit": "warp-instructions/s", "frac": round(achieved / peak, 4),
            "instructions_per_launch": int(inst), "sm_mhz": mhz, "sms": sms}


# ------------------------------------------------------------ CPU oracle

def oracle_sample(name: str, bits, nthreads: int = 0):
    """Encode + decode a bounded sample (bits = the first tokens of the
    workload) with the CPU oracle on nthreads host cores (0: all). Returns
    (seconds, raw bytes, threads, encoded)."""
    from oracle import oracle
    p, k, v = workload_info(name)
    L, _, T, C = bits.shape
    ch = p["chunk_tokens"][0]
    nth = nthreads if nthreads > 0 else oracle.max_threads()
    t0 = time.perf_counter()
    enc = oracle.encode(bits, ch, k, v, nthreads=nth)
    oracle.decode(enc, L, T, C, ch, k, v, nthreads=nth)
    dt = time.perf_counter() - t0
    return dt, bits.nbytes, nth, enc


def cpu_baseline(name: str, tokens: int):
    """The oracle on all host cores over the first `tokens` tokens, and on one
    core over a sixteenth of them."""
    from kv_cache_compression_03_gb300 import synthetic
    bits = synthetic.generate(name, num_tokens=tokens)
    dt, raw, nth, _ = oracle_sample(name, bits)
    t1 = max(1, tokens // 16)
    dt1, raw1, _, _ = oracle_sample(name, bits[:, :, :t1].copy(), nthreads=1)
    p, _, _ = workload_info(name)
    return {"value": round(raw / dt / 1e9, 4), "unit": "GB/s", "cores": nth, "kind": "oracle",
            "sample": f"first {tokens} of {p['T']} tokens, all {p['L']} layers, K and V "
                      f"({raw / 1e6:.1f} MB raw bf16), encode+decode, {dt:.2f} s wall",
            "single_core": {"value": round(raw1 / dt1 / 1e9, 4), "unit": "GB/s",
                            "sample": f"first {t1} tokens ({raw1 / 1e6:.1f} MB), "
                                      f"{dt1:.2f} s wall"}}


def run_reference(args):
    rank, world, _ = dist_env()
    if world > 1 and rank != 0:
        return 0
    from kv_cache_compression_03_gb300 import synthetic
    p, _, _ = workload_info(args.workload)
    tokens = args.cpu_tokens
    bits = synthetic.generate(args.workload, num_tokens=tokens)
    for _ in range(args.warmup):
        oracle_sample(args.workload, bits)
    times = []
    raw = 0
    nth = 1
    for _ in range(args.steps):
        dt, raw, nth, _ = oracle_sample(args.workload, bits)
        times.append(dt)
    tot = sum(times)
    value = raw * len(times) / tot / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * tot / len(times), 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": args.workload, "layers": p["L"], "tokens": p["T"],
                   "kv_heads": p["H"], "head_size": p["D"], "chunk_tokens": p["chunk_tokens"][0],
                   "sample_tokens": tokens, "device": "host cores (CPU oracle)"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": nth,
                         "kind": "oracle",
                         "sample": f"first {tokens} of {p['T']} tokens per step, encode+decode"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0, "clocks": None,
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ GPU

def rel_rmse(x, y) -> float:
    """||y - x|| / ||x|| over a whole bf16 blob, one layer at a time."""
    num = den = 0.0
    for l in range(x.shape[0]):
        xf = x[l].float()
        num += float((y[l].float() - xf).pow(2).sum())
        den += float(xf.pow(2).sum())
    return (num / den) ** 0.5 if den > 0 else 0.0


TRANSFER_MBPS = (100, 500, 1000)


def transfer_model(raw: int, sizes: dict, decode_ms: dict):
    """Seconds to move one blob over a link of 100/500/1000 Mbit/s and
    decode it: bytes * 8 / bandwidth, plus the measured GPU decode time
    (none for raw bf16)."""
    out = {"bandwidth_mbps": list(TRANSFER_MBPS)}
    for key, nbytes in [("raw", raw)] + list(sizes.items()):
        dec_s = decode_ms.get(key, 0.0) * 1e-3
        out[key + "_s"] = [round(nbytes * 8 / (bw * 1e6) + dec_s, 4) for bw in TRANSFER_MBPS]
    return out


def measure_baselines(cg, kv, cg_out, raw, container, t_dec_ms, peak, stream, dev, args):
    """The comparison codecs on the same input, after the timed region: the
    int8 + per-row-scale codec (its own encode and decode loops, CUDA events
    on the launch stream) and naive serialisation (the raw bytes); the
    reconstruction error of each lossy codec; and the transfer-time model."""
    import torch
    L, _, T, H, D = kv.shape
    C = H * D
    rows = 2 * L * T
    q = torch.empty(rows * C, dtype=torch.int8, device=dev)
    scales = torch.empty(rows, dtype=torch.float32, device=dev)
    status = torch.empty(16, dtype=torch.uint8, device=dev)
    y = torch.empty_like(kv)

    def enc8():
        cg.cg_int8_encode(kv, rows, C, q, scales, status, stream)

    def dec8():
        cg.cg_int8_decode(q, scales, rows, C, y, stream)

    for _ in range(max(args.warmup, 1)):
        enc8()
        dec8()
    st, _ = cg.cg_last_device_error(None, status, stream)
    assert st == cg.CG_OK, st
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    torch.cuda.synchronize(dev)
    ev[0].record(stream)
    for _ in range(args.steps):
        enc8()
    ev[1].record(stream)
    for _ in range(args.steps):
        dec8()
    ev[2].record(stream)
    torch.cuda.synchronize(dev)
    t_e = ev[0].elapsed_time(ev[1]) / args.steps
    t_d = ev[1].elapsed_time(ev[2]) / args.steps
    int8_bytes = rows * C + 4 * rows
    alg = raw + int8_bytes
    int8 = {"encode_gbs": round(raw / (t_e * 1e-3) / 1e9, 2),
            "decode_gbs": round(raw / (t_d * 1e-3) / 1e9, 2),
            "encode_ms": round(t_e, 4), "decode_ms": round(t_d, 4),
            "encode_hbm_frac": round(alg / (t_e * 1e-3) / 1e9 / peak, 4),
            "decode_hbm_frac": round(alg / (t_d * 1e-3) / 1e9 / peak, 4),
            "compression_ratio": round(raw / int8_bytes, 4), "bytes": int(int8_bytes),
            "rel_rmse": round(rel_rmse(kv, y), 6),
            "kernels": ["k_int8_encode", "k_int8_decode"]}
    return {
        "int8": int8,
        "naive": {"compression_ratio": 1.0, "bytes": int(raw), "rel_rmse": 0.0},
        "cachegen": {"compression_ratio": round(raw / container, 4), "bytes": int(container),
                     "rel_rmse": round(rel_rmse(kv, cg_out), 6)},
        "transfer_model": transfer_model(raw, {"cachegen": container, "int8": int8_bytes},
                                         {"cachegen": t_dec_ms, "int8": t_d}),
    }


def sweep_settings(L: int):
    """Bin settings of the sweep: the preset, then every layer at 8, 16, 32
    and 64 bins, then the preset with its 32-bin ranges widened (K's first
    L/2 layers, V's first 10)."""
    from kv_cache_compression_03_gb300 import cachegen as cg
    k, v = cg.preset_specs(L)
    out = [("preset", k, v)]
    for b in (8, 16, 32, 64):
        out.append((f"uniform{b}", [(0, L, b)], [(0, L, b)]))
    if L >= 20:
        out.append(("preset_wide32", [(0, L // 2, 32), (L // 2, L, 16)],
                    [(0, 10, 32), (10, L, 16)]))
    return out


def run_bins_sweep(args):
    """Compression ratio against reconstruction error for several bin
    settings on one workload: one JSON line per setting (device-timed
    encode and decode over --steps steps)."""
    import numpy as np
    import torch

    from kv_cache_compression_03_gb300 import cachegen as cg
    from kv_cache_compression_03_gb300 import synthetic

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    name = args.workload
    p, _, _ = workload_info(name)
    L, T, H, D = p["L"], (args.tokens or p["T"]), p["H"], p["D"]
    ch = p["chunk_tokens"][0]
    bits = synthetic.generate(name, num_tokens=T)
    kv = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).reshape(L, 2, T, H, D).to(dev)
    del bits
    stream = torch.cuda.current_stream(dev)
    for label, k, v in sweep_settings(L):
        try:
            codec = cg.Codec(L, T, H, D, ch, k, v, device=dev)
        except cg.CacheGenError as e:
            print(json.dumps({"sweep": "bins", "workload": name, "setting": label,
                              "unavailable": str(e)}), flush=True)
            continue
        enc = codec.encode(kv)
        out = codec.decode(enc)
        raw = codec.sizes.raw_bytes
        container = cg.cg_container_size(codec.plan, enc.stream_bytes)
        for _ in range(args.warmup):
            codec.encode(kv, enc, sync=False, stream=stream)
            codec.decode(enc, out, sync=False, stream=stream)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        torch.cuda.synchronize(dev)
        ev[0].record(stream)
        for _ in range(args.steps):
            codec.encode(kv, enc, sync=False, stream=stream)
        ev[1].record(stream)
        for _ in range(args.steps):
            codec.decode(enc, out, sync=False, stream=stream)
        ev[2].record(stream)
        torch.cuda.synchronize(dev)
        st, _ = cg.cg_last_device_error(codec.plan, codec.workspace)
        assert st == cg.CG_OK, st
        t_e = ev[0].elapsed_time(ev[1]) / args.steps
        t_d = ev[1].elapsed_time(ev[2]) / args.steps
        line = {"sweep": "bins", "workload": name, "tokens": T, "setting": label,
                "kspecs": [list(s) for s in k], "vspecs": [list(s) for s in v],
                "compression_ratio": round(raw / container, 4),
                "stream_bits_per_value": round(8 * enc.stream_bytes / (raw / 2), 4),
                "rel_rmse": round(rel_rmse(kv, out), 6),
                "rel_rmse_k": round(rel_rmse(kv[:, 0:1], out[:, 0:1]), 6),
                "rel_rmse_v": round(rel_rmse(kv[:, 1:2], out[:, 1:2]), 6),
                "encode_gbs": round(raw / (t_e * 1e-3) / 1e9, 2),
                "decode_gbs": round(raw / (t_d * 1e-3) / 1e9, 2)}
        print(json.dumps(line), flush=True)
        del codec, enc, out
    return 0


def run_chunk_sweep(args):
    """The chunk-size sweep workload: for each chunk_tokens, encode and decode
    timed separately (device events), the ratio of the whole-blob container
    and of the per-object containers, and the time to write all per-object
    containers. One JSON line per chunk size."""
    import numpy as np
    import torch

    from kv_cache_compression_03_gb300 import cachegen as cg
    from kv_cache_compression_03_gb300 import synthetic

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    name = "mistral7b_chunk_sweep"
    p, k, v = workload_info(name)
    L, T, H, D = p["L"], p["T"], p["H"], p["D"]
    bits = synthetic.generate(name)
    kv = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).reshape(L, 2, T, H, D).to(dev)
    stream = torch.cuda.current_stream(dev)
    for ch in p["chunk_tokens"]:
        codec = cg.Codec(L, T, H, D, ch, k, v, device=dev)
        enc = codec.encode(kv)
        out = codec.decode(enc)
        raw = codec.sizes.raw_bytes
        container = cg.cg_container_size(codec.plan, enc.stream_bytes)
        for _ in range(args.warmup):
            codec.encode(kv, enc, sync=False, stream=stream)
            codec.decode(enc, out, sync=False, stream=stream)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        torch.cuda.synchronize(dev)
        ev[0].record(stream)
        for _ in range(args.steps):
            codec.encode(kv, enc, sync=False, stream=stream)
        ev[1].record(stream)
        for _ in range(args.steps):
            codec.decode(enc, out, sync=False, stream=stream)
        ev[2].record(stream)
        torch.cuda.synchronize(dev)
        st, _ = cg.cg_last_device_error(codec.plan, codec.workspace)
        assert st == cg.CG_OK, st
        t_e = ev[0].elapsed_time(ev[1]) / args.steps
        t_d = ev[1].elapsed_time(ev[2]) / args.steps
        t0 = time.perf_counter()
        objs = codec.object_bytes(enc)
        t_obj = time.perf_counter() - t0
        obj_bytes = sum(int(o.numel()) for o in objs)
        line = {"sweep": "chunk_tokens", "workload": name, "tokens": T, "chunk_tokens": ch,
                "groups": codec.sizes.num_groups, "objects": len(objs),
                "encode_gbs": round(raw / (t_e * 1e-3) / 1e9, 2),
                "decode_gbs": round(raw / (t_d * 1e-3) / 1e9, 2),
                "encode_ms": round(t_e, 4), "decode_ms": round(t_d, 4),
                "compression_ratio": round(raw / container, 4),
                "per_object_ratio": round(raw / obj_bytes, 4),
                "per_object_serialize_ms": round(1e3 * t_obj, 3),
                "l2": "the whole blob (%.1f MB) fits in L2" % (raw / 1e6)}
        print(json.dumps(line), flush=True)
        del codec, enc, out
    return 0


def run_codec(args):
    import numpy as np
    import torch

    from kv_cache_compression_03_gb300 import cachegen as cg
    from kv_cache_compression_03_gb300 import synthetic

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    name = args.workload
    p, k, v = workload_info(name)
    L, T, H, D = p["L"], (args.tokens or p["T"]), p["H"], p["D"]
    C = H * D
    ch = p["chunk_tokens"][0]

    # CPU baseline first (before any heavy GPU work; OpenMP threads only)
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(name, args.cpu_tokens)

    bits = synthetic.generate(name, num_tokens=T)
    host_kv = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).reshape(L, 2, T, H, D)
    kv = host_kv.to(dev)
    codec = cg.Codec(L, T, H, D, ch, k, v, device=dev)
    sizes = codec.sizes
    raw = sizes.raw_bytes
    enc = codec.alloc_encoded()
    out = torch.empty_like(kv)
    stream = torch.cuda.current_stream(dev)

    def step():
        cg.cg_encode(codec.plan, kv, codec.workspace, enc.bytestream, enc.lengths, enc.cdf,
                     enc.amax, stream)
        cg.cg_decode(codec.plan, enc.bytestream, enc.lengths, enc.cdf, enc.amax,
                     enc.stream_bytes, codec.workspace, out, stream)

    # one checked encode to learn the stream size
    codec.encode(kv, enc)
    st, total = cg.cg_last_device_error(codec.plan, codec.workspace)
    assert st == cg.CG_OK, st
    enc.stream_bytes = total
    container = cg.cg_container_size(codec.plan, total)
    for _ in range(max(args.warmup, 1)):
        step()
    st, _ = cg.cg_last_device_error(codec.plan, codec.workspace)
    assert st == cg.CG_OK, st
    torch.cuda.synchronize(dev)

    launches_per_step = sizes.encode_launches + sizes.decode_launches
    cg.cg_profile_enable(codec.plan, launches_per_step * args.steps + 8)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize(dev)
    with ClockSampler(dev.index if dev.index is not None else 0) as clk:
        e0.record(stream)
        for _ in range(args.steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize(dev)
    barrier(world)
    ms_local = e0.elapsed_time(e1)
    prof = cg.cg_profile_read(codec.plan)
    cg.cg_profile_enable(codec.plan, 0)
    st, _ = cg.cg_last_device_error(codec.plan, codec.workspace)
    assert st == cg.CG_OK, st
    ms_total = aggregate_max(ms_local, world, dev)
    ms_step = ms_total / args.steps
    value = world * raw * args.steps / (ms_total * 1e-3) / 1e9

    enc_names = ("k_encode_tiles", "k_scan_tiles(encode)", "k_pack")
    dec_names = ("k_tile_sums", "k_scan_tiles(decode)", "k_decode_tiles")
    t_enc = sum(prof[n][1] for n in enc_names if n in prof) / args.steps
    t_dec = sum(prof[n][1] for n in dec_names if n in prof) / args.steps

    # dominant kernel and its roofline
    top = max(prof.items(), key=lambda kv_: kv_[1][1])
    kname, (klaunch, kms) = top
    side_bytes = 4 * sizes.num_scales + 4 * sizes.num_streams + 2 * sizes.cdf_entries
    alg_bytes = raw + side_bytes + total     # read raw, write all sections (or the reverse)
    per_launch_ms = kms / klaunch
    achieved = alg_bytes / (per_launch_ms * 1e-3) / 1e9
    peak, peak_kind = peaks()
    full_size = (T == p["T"])  # the recorded counters are per full-size launch
    traffic = recorded_counter(kname, name) if full_size else None
    roof = {"kernel": kname, "bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
            "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": traffic,
            "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
            else "fallback 6.8 TB/s", "algorithmic_bytes_per_launch": int(alg_bytes),
            "ms_per_launch": round(per_launch_ms, 4)}

    # end to end through host buffers, streamed by layer groups: every group of
    # G layers is a CacheGen blob of its own (contiguous in host memory, its own
    # plan; its tiles code exactly as in the whole blob). Each group uploads and
    # encodes on one of three rotating streams while the host serialises and
    # deserialises the group before it, whose decode and download then run on
    # its own stream; every step copies the whole blob up and its result back.
    e2e = None
    if not args.no_e2e:
        host_in = torch.empty_like(host_kv, device="cpu").pin_memory()
        host_in.copy_(host_kv)
        host_out = torch.empty_like(host_in).pin_memory()
        n_e2e = max(2, min(args.steps, 6))
        G = 4 if L % 4 == 0 else 1

        def slice_specs(specs, l0, l1):
            return [(max(a, l0) - l0, min(b, l1) - l0, bins) for a, b, bins in specs
                    if a < l1 and b > l0]

        streams = [torch.cuda.Stream(dev) for _ in range(3)]
        parts = []
        for l0 in range(0, L, G):
            l1 = min(l0 + G, L)
            c = cg.Codec(l1 - l0, T, H, D, ch, slice_specs(k, l0, l1), slice_specs(v, l0, l1),
                         device=dev)
            parts.append({
                "l0": l0, "l1": l1, "codec": c, "stream": streams[len(parts) % 3],
                "kv": torch.empty_like(kv[l0:l1]), "out": torch.empty_like(kv[l0:l1]),
                "enc": c.alloc_encoded(), "enc2": c.alloc_encoded(),
                "blob": torch.empty(cg.cg_container_size(c.plan, c.sizes.max_stream_bytes),
                                    dtype=torch.uint8).pin_memory()})

        def head(pt):
            c, st, e = pt["codec"], pt["stream"], pt["enc"]
            with torch.cuda.stream(st):
                pt["kv"].copy_(host_in[pt["l0"]:pt["l1"]], non_blocking=True)
                cg.cg_encode(c.plan, pt["kv"], c.workspace, e.bytestream, e.lengths, e.cdf,
                             e.amax, st)

        def tail(pt):
            c, st, e, e2 = pt["codec"], pt["stream"], pt["enc"], pt["enc2"]
            with torch.cuda.stream(st):
                code, sb = cg.cg_last_device_error(c.plan, c.workspace, st)
                n = cg.cg_serialize(c.plan, e.bytestream, e.lengths, e.cdf, e.amax, sb,
                                    pt["blob"], st)
                cg.cg_deserialize(c.plan, pt["blob"][:n], e2.bytestream, e2.lengths, e2.cdf,
                                  e2.amax, st)
                cg.cg_decode(c.plan, e2.bytestream, e2.lengths, e2.cdf, e2.amax, sb,
                             c.workspace, pt["out"], st)
                host_out[pt["l0"]:pt["l1"]].copy_(pt["out"], non_blocking=True)
            return code, n

        def e2e_step():
            res = []
            head(parts[0])
            for i, pt in enumerate(parts):
                if i + 1 < len(parts):
                    head(parts[i + 1])
                res.append(tail(pt))
            return res

        e2e_step()
        torch.cuda.synchronize(dev)
        # three timed runs of n_e2e steps; the figure is their median (the
        # host link and the host's memory are shared with other tenants, and
        # single runs have read far below the others)
        runs = []
        for _ in range(3):
            barrier(world)
            t0 = time.perf_counter()
            for _ in range(n_e2e):
                res = e2e_step()
            torch.cuda.synchronize(dev)
            t_e2e = aggregate_max(time.perf_counter() - t0, world, dev)
            runs.append(world * raw * n_e2e / t_e2e / 1e9)
            assert all(code == cg.CG_OK for code, _ in res)
        assert torch.equal(host_out.view(torch.int16), out.view(torch.int16).cpu())
        blob_bytes = sum(n for _, n in res)
        e2e = {"value": round(sorted(runs)[1], 3), "unit": "GB/s",
               "runs": [round(r, 3) for r in runs], "statistic": "median of 3 runs",
               "h2d_bytes_per_step": int(raw + blob_bytes),
               "d2h_bytes_per_step": int(blob_bytes + raw), "steps": n_e2e,
               "path": f"pinned host kv -> per {G}-layer group: H2D -> cg_encode -> "
               "cg_serialize (D2H container) -> cg_deserialize (H2D) -> cg_decode -> D2H; "
               "groups pipelined on three streams"}
        del parts

    baselines = None
    if not args.no_baselines:
        baselines = measure_baselines(cg, kv, out, raw, container, t_dec, peak, stream, dev, args)

    if rank != 0:
        return 0
    clocks = clk.summary()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    issue = issue_ceiling(kname, name if full_size else "", per_launch_ms, sms,
                          (clocks or {}).get("sm_max_mhz"))
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": name, "layers": L, "tokens": T, "kv_heads": H, "head_size": D,
                   "chunk_tokens": ch, "group_tokens": 256,
                   "bins": {"k": [list(s) for s in k], "v": [list(s) for s in v]},
                   "l2": "inputs larger than L2 (raw KV per step %.2f GB)" % (raw / 1e9),
                   "parallelism": f"replicas x{world}"},
        "encode_gbs": round(raw / (t_enc * 1e-3) / 1e9, 2),
        "decode_gbs": round(raw / (t_dec * 1e-3) / 1e9, 2),
        "encode_hbm_frac": round((raw + side_bytes + total) / (t_enc * 1e-3) / 1e9 / peak, 4),
        "decode_hbm_frac": round((raw + side_bytes + total) / (t_dec * 1e-3) / 1e9 / peak, 4),
        "compression_ratio": round(raw / container, 4),
        "stream_bits_per_value": round(8 * total / (raw / 2), 4),
        "container_bytes": int(container),
        "kernels": {n: {"launches": c, "ms_per_launch": round(ms / c, 4)}
                    for n, (c, ms) in prof.items()},
        "roofline": roof,
        "issue": issue,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "baselines": baselines,
        "clocks": clocks,
        "gpu_launches": int(launches_per_step * args.steps),
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["cachegen", "reference"], default="cachegen")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--tokens", type=int, default=None,
                    help="truncate the workload to this many tokens (profiling runs)")
    ap.add_argument("--cpu-tokens", type=int, default=2048,
                    help="tokens of the workload in the CPU oracle's bounded sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-baselines", action="store_true",
                    help="skip the int8/naive comparison codecs and the transfer-time model")
    ap.add_argument("--sweep-bins", action="store_true",
                    help="instead of the benchmark line: ratio vs reconstruction error for "
                         "several bin settings, one JSON line each")
    ap.add_argument("--sweep-chunks", action="store_true",
                    help="instead of the benchmark line: the chunk-size sweep workload, "
                         "one JSON line per chunk_tokens")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.sweep_bins:
        return run_bins_sweep(args)
    if args.sweep_chunks:
        return run_chunk_sweep(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_codec(args)


if __name__ == "__main__":
    sys.exit(main())
