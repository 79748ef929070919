"""Seeded synthetic KV caches shaped like the codec's workloads.

This module only draws inputs: it holds none of the codec's arithmetic, and
both the CUDA path's tests and the CPU oracle consume what it returns.

Value model (per K/V and layer, each with its own generator spawned from
the workload seed): a per-channel scale sigma_c ~ LogNormal(0, s), a few
K-channel outliers multiplied by a constant, and an AR(1) process along
tokens, x_0 = sigma z_0, x_t = rho x_{t-1} + sqrt(1 - rho^2) sigma z_t,
with z standard normal or a unit-variance Student-t. The long-context
workload also scales 1 % of the tokens (the same token indices for every
layer and for K and V) by 5. Values are rounded fp32 -> bf16 (nearest
even) and returned as uint16 bit patterns, laid out [L, 2, T, H*D].

The shapes follow the models the CacheGen pages name: OPT-125m, a 7B
(Mistral/Llama-3.1-8B, 32 layers x 8 KV heads x 128) cache at 1K and 16K
tokens, the chunk-size sweep of LMCache's benchmark (32 x 8 x 128, chunk
64/128/256/768), and GLM-4-9B (40 layers x 2 KV heads x 128).
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

# Bin specs per [start_layer, end_layer): K's first 10 layers and V's first
# 2 layers use 32 bins, the rest 16 (the 7B/8B/9B presets; OPT-125m's 12
# layers follow the same rule).
def _spec_10_2(L):
    k = [(0, min(10, L), 32)] + ([(10, L, 16)] if L > 10 else [])
    v = [(0, min(2, L), 32)] + ([(2, L, 16)] if L > 2 else [])
    return k, v


WORKLOADS = {
    "opt125m_t256": dict(L=12, T=256, H=12, D=64, chunk_tokens=(256,), dist="normal",
                         sigma_ln=0.5, rho=0.9, n_outlier=4, outlier_scale=10.0,
                         spike_frac=0.0, spike=1.0, seed=1001),
    "mistral7b_t1k": dict(L=32, T=1024, H=8, D=128, chunk_tokens=(256,), dist="normal",
                          sigma_ln=0.5, rho=0.9, n_outlier=4, outlier_scale=10.0,
                          spike_frac=0.0, spike=1.0, seed=1002),
    "mistral7b_chunk_sweep": dict(L=32, T=768, H=8, D=128, chunk_tokens=(64, 128, 256, 768),
                                  dist="normal", sigma_ln=0.5, rho=0.9, n_outlier=4,
                                  outlier_scale=10.0, spike_frac=0.0, spike=1.0, seed=1003),
    "llama8b_t16k": dict(L=32, T=16384, H=8, D=128, chunk_tokens=(256,), dist="student_t4",
                         sigma_ln=0.5, rho=0.9, n_outlier=4, outlier_scale=10.0,
                         spike_frac=0.01, spike=5.0, seed=1004),
    "glm4_9b_t32k": dict(L=40, T=32768, H=2, D=128, chunk_tokens=(256,), dist="normal",
                         sigma_ln=1.0, rho=0.95, n_outlier=8, outlier_scale=20.0,
                         spike_frac=0.0, spike=1.0, seed=1005),
}


def workload_specs(name: str):
    """(kspecs, vspecs) of a workload: lists of (start, end, bins)."""
    return _spec_10_2(WORKLOADS[name]["L"])


def _to_bf16_bits(x: np.ndarray) -> np.ndarray:
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def _ar1(e: np.ndarray, rho: float) -> np.ndarray:
    """x_t = rho x_{t-1} + e_t along axis 0 (x_{-1} = 0)."""
    try:
        from scipy.signal import lfilter
        return lfilter([1.0], [1.0, -rho], e, axis=0)
    except ImportError:  # plain loop fallback
        x = np.empty_like(e)
        acc = np.zeros(e.shape[1:], dtype=e.dtype)
        for t in range(e.shape[0]):
            acc = rho * acc + e[t]
            x[t] = acc
        return x


def _draw_layer(ss: np.random.SeedSequence, T: int, C: int, is_k: bool, p: dict,
                spike_rows, out: np.ndarray):
    rng = np.random.Generator(np.random.PCG64(ss))
    sigma = rng.lognormal(0.0, p["sigma_ln"], C)
    if is_k and p["n_outlier"] > 0:
        idx = rng.choice(C, p["n_outlier"], replace=False)
        sigma[idx] *= p["outlier_scale"]
    if p["dist"] == "student_t4":
        z = rng.standard_t(4.0, (T, C)) / math.sqrt(2.0)
    else:
        z = rng.standard_normal((T, C))
    rho = p["rho"]
    z[1:] *= math.sqrt(1.0 - rho * rho)
    x = _ar1(z, rho)
    x *= sigma[None, :]
    if spike_rows is not None:
        x[spike_rows] *= p["spike"]
    out[...] = _to_bf16_bits(x)


def generate(name: str, num_tokens: int | None = None, threads: int | None = None) -> np.ndarray:
    """Return the workload's KV as uint16 bf16 bits shaped [L, 2, T, H*D].

    ``num_tokens`` truncates (or extends) the token axis while keeping the
    value model, for reduced-size cases."""
    p = WORKLOADS[name]
    L, H, D = p["L"], p["H"], p["D"]
    T = p["T"] if num_tokens is None else int(num_tokens)
    C = H * D
    root = np.random.SeedSequence(p["seed"])
    children = root.spawn(2 * L + 1)
    spike_rows = None
    if p["spike_frac"] > 0:
        srng = np.random.Generator(np.random.PCG64(children[2 * L]))
        nspk = max(1, int(round(p["spike_frac"] * T)))
        spike_rows = np.sort(srng.choice(T, nspk, replace=False))
    kv = np.empty((L, 2, T, C), dtype=np.uint16)
    jobs = [(kvs, l) for kvs in range(2) for l in range(L)]
    nthreads = threads or min(16, os.cpu_count() or 1)

    def run(job):
        kvs, l = job
        _draw_layer(children[kvs * L + l], T, C, kvs == 0, p, spike_rows, kv[l, kvs])

    if nthreads > 1:
        with ThreadPoolExecutor(nthreads) as ex:
            list(ex.map(run, jobs))
    else:
        for j in jobs:
            run(j)
    return kv


def random_kv(L: int, T: int, C: int, seed: int, scale: float = 1.0) -> np.ndarray:
    """Plain i.i.d. normal KV of any shape (for edge cases), bf16 bits."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return _to_bf16_bits(rng.standard_normal((L, 2, T, C)) * scale)
