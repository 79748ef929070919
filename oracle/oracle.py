"""Python access to the CPU oracle (``cachegen_oracle.c``).

TEST INFRASTRUCTURE. Only the tests, the package smoke check and the bench's
CPU-baseline leg import this module; the codec's product path never does.
It shares no code with the CUDA path: it compiles and loads its own C file.

Arrays are numpy: bf16 values travel as their uint16 bit patterns.
Specs are lists of ``(start_layer, end_layer, bins)`` with ``[start, end)``
layer ranges ("LMCache 中的 KV Cache 压缩：CacheGen 编解码原理、配置方式与源码解析",
§1 QuantizationSpec).
"""
from __future__ import annotations

import ctypes as ct
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "cachegen_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libcgoracle.so")

OK, ERR_INVALID_ARG, ERR_SPEC, ERR_CAPACITY, ERR_NONFINITE, ERR_CORRUPT = 0, 1, 2, 3, 4, 5

_lock = threading.Lock()
_lib = None


class OracleError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"oracle {what} failed with status {status}")
        self.status = status


def compile_source(src: str, out: str) -> None:
    """Compile a C file with the oracle's flags (no OpenMP)."""
    subprocess.run(["gcc", "-O2", "-std=c99", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
                    "-shared", "-o", out, src, "-lm"], check=True, capture_output=True)


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP when available). Returns the .so path.

    ``CG_ORACLE_LIB`` names a prebuilt library to load instead (the mutation
    tests use it to load deliberately broken copies)."""
    override = os.environ.get("CG_ORACLE_LIB")
    if override:
        return override
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    base = ["gcc", "-O2", "-std=c99", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    try:
        subprocess.run(base + ["-fopenmp", "-o", tmp, _SRC, "-lm"], check=True,
                       capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base + ["-o", tmp, _SRC, "-lm"], check=True, capture_output=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib() -> ct.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            path = build()
            L = ct.CDLL(path)
            P = ct.c_void_p
            i32, i64, sz = ct.c_int32, ct.c_int64, ct.c_size_t
            sig = {
                "orc_layer_bins": (ct.c_int, [i32, P, i32, P]),
                "orc_groups": (i32, [i32, i32, P, P]),
                "orc_num_groups": (i32, [i32, i32]),
                "orc_quantize_row": (ct.c_int, [P, i32, i32, P, P]),
                "orc_dequant_row": (None, [P, i32, i32, ct.c_float, P]),
                "orc_int_cdf": (None, [P, i32, ct.c_uint32, P]),
                "orc_wnc_encode": (ct.c_int, [P, i32, P, i32, i32, P, sz, P]),
                "orc_wnc_decode": (ct.c_int, [P, sz, i32, P, i32, i32, P]),
                "orc_cdf_entries": (i64, [i32, i32, i32, i32, P, i32, P, i32]),
                "orc_encode": (ct.c_int, [P, i32, i32, i32, i32, P, i32, P, i32, P, P, P, P, sz,
                                          P, P, i32]),
                "orc_decode": (ct.c_int, [P, sz, P, P, P, i32, i32, i32, i32, P, i32, P, i32, P,
                                          P, i32]),
                "orc_encode_tiles": (ct.c_int, [P, i32, i32, i32, i32, P, i32, P, i32, P, i32, P,
                                                P, P, P, sz, P, i32]),
                "orc_container_size": (i64, [i32, i32, i32, i64, i64]),
                "orc_serialize": (ct.c_int, [i32, i32, i32, i32, i32, P, i32, P, i32, P, P, P, i64,
                                             P, i64, P, i64]),
                "orc_max_threads": (i32, []),
                "orc_int8_quantize_row": (ct.c_int, [P, i32, P, P]),
                "orc_int8_dequant_row": (None, [P, i32, ct.c_float, P]),
                "orc_int8_encode": (ct.c_int, [P, i64, i32, P, P, i32]),
                "orc_int8_decode": (None, [P, P, i64, i32, P, i32]),
            }
            for name, (res, args) in sig.items():
                f = getattr(L, name)
                f.restype = res
                f.argtypes = args
            _lib = L
    return _lib


def _p(a: np.ndarray):
    return a.ctypes.data_as(ct.c_void_p)


def _specs(specs) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(specs, dtype=np.int32).reshape(-1, 3))


def _check(st: int, what: str):
    if st != OK:
        raise OracleError(st, what)


def max_threads() -> int:
    return int(lib().orc_max_threads())


# ---------------------------------------------------------------- config

def layer_bins(num_layers: int, specs) -> np.ndarray:
    s = _specs(specs)
    out = np.zeros(num_layers, dtype=np.int32)
    _check(lib().orc_layer_bins(num_layers, _p(s), len(s), _p(out)), "layer_bins")
    return out


def groups(num_tokens: int, chunk_tokens: int):
    n = lib().orc_num_groups(num_tokens, chunk_tokens)
    if n < 0:
        raise OracleError(ERR_INVALID_ARG, "groups")
    start = np.zeros(n, dtype=np.int32)
    count = np.zeros(n, dtype=np.int32)
    lib().orc_groups(num_tokens, chunk_tokens, _p(start), _p(count))
    return start, count


# ------------------------------------------------------ per-row / per-stream

def quantize_row(x_bits: np.ndarray, bins: int):
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    q = np.zeros(x.size, dtype=np.uint8)
    a = ct.c_float(0.0)
    _check(lib().orc_quantize_row(_p(x), x.size, bins, ct.byref(a), _p(q)), "quantize_row")
    return float(np.float32(a.value)), q


def dequant_row(q: np.ndarray, bins: int, amax: float) -> np.ndarray:
    q = np.ascontiguousarray(q, dtype=np.uint8)
    y = np.zeros(q.size, dtype=np.uint16)
    lib().orc_dequant_row(_p(q), q.size, bins, ct.c_float(amax), _p(y))
    return y


def int_cdf(count: np.ndarray, n: int) -> np.ndarray:
    c = np.ascontiguousarray(count, dtype=np.uint32)
    out = np.zeros(c.size + 1, dtype=np.uint32)
    lib().orc_int_cdf(_p(c), c.size, n, _p(out))
    return out


def wnc_encode(sym: np.ndarray, cdf_rows: np.ndarray) -> bytes:
    """Encode symbols; cdf_rows[i] is the (N+1)-entry CDF used for symbol i."""
    s = np.ascontiguousarray(sym, dtype=np.uint8)
    rows = np.ascontiguousarray(cdf_rows, dtype=np.uint32)
    if rows.ndim == 1:
        rows = np.ascontiguousarray(np.broadcast_to(rows, (s.size, rows.size)))
    N = rows.shape[1] - 1
    cap = 2 * s.size + 8
    out = np.zeros(cap, dtype=np.uint8)
    nb = ct.c_size_t(0)
    _check(lib().orc_wnc_encode(_p(s), s.size, _p(rows), rows.shape[1], N, _p(out), cap,
                                ct.byref(nb)), "wnc_encode")
    return out[: nb.value].tobytes()


def wnc_decode(data: bytes, nsym: int, cdf_rows: np.ndarray) -> np.ndarray:
    rows = np.ascontiguousarray(cdf_rows, dtype=np.uint32)
    if rows.ndim == 1:
        rows = np.ascontiguousarray(np.broadcast_to(rows, (nsym, rows.size)))
    N = rows.shape[1] - 1
    buf = np.frombuffer(bytes(data) + b"\0", dtype=np.uint8).copy()
    out = np.zeros(nsym, dtype=np.uint8)
    _check(lib().orc_wnc_decode(_p(buf), len(data), nsym, _p(rows), rows.shape[1], N, _p(out)),
           "wnc_decode")
    return out


# -------------------------------------------------------------- whole blob

def cdf_entries(L, T, C, chunk_tokens, kspecs, vspecs) -> int:
    k, v = _specs(kspecs), _specs(vspecs)
    e = lib().orc_cdf_entries(L, T, C, chunk_tokens, _p(k), len(k), _p(v), len(v))
    if e < 0:
        raise OracleError(ERR_SPEC, "cdf_entries")
    return int(e)


def encode(kv_bits: np.ndarray, chunk_tokens: int, kspecs, vspecs, nthreads: int = 0,
           want_symbols: bool = False) -> dict:
    """Encode kv_bits[L, 2, T, C] (uint16 bf16 bits; a [L,2,T,H,D] array is
    flattened over heads). Returns amax, cdf, lengths, stream bytes and
    optionally the symbols."""
    kv = np.ascontiguousarray(kv_bits, dtype=np.uint16)
    L, two, T = kv.shape[:3]
    assert two == 2
    C = int(np.prod(kv.shape[3:]))
    k, v = _specs(kspecs), _specs(vspecs)
    ent = cdf_entries(L, T, C, chunk_tokens, k, v)
    amax = np.zeros((2, L, T), dtype=np.float32)
    cdf = np.zeros(ent, dtype=np.uint16)
    lengths = np.zeros(2 * L * T, dtype=np.int32)
    cap = 2 * L * T * (2 * C + 2)
    out = np.zeros(cap, dtype=np.uint8)
    sym = np.zeros((2, L, T, C), dtype=np.uint8) if want_symbols else None
    total = ct.c_size_t(0)
    nth = nthreads if nthreads > 0 else max_threads()
    _check(lib().orc_encode(_p(kv), L, T, C, chunk_tokens, _p(k), len(k), _p(v), len(v),
                            _p(amax), _p(cdf), _p(lengths), _p(out), cap, ct.byref(total),
                            _p(sym) if sym is not None else None, nth), "encode")
    res = {"amax": amax, "cdf": cdf, "lengths": lengths,
           "bytes": out[: total.value].copy(), "stream_bytes": int(total.value)}
    if sym is not None:
        res["symbols"] = sym
    return res


def decode(enc: dict, L: int, T: int, C: int, chunk_tokens: int, kspecs, vspecs,
           nthreads: int = 0, want_symbols: bool = False):
    k, v = _specs(kspecs), _specs(vspecs)
    data = np.ascontiguousarray(enc["bytes"], dtype=np.uint8)
    if data.size == 0:
        data = np.zeros(1, dtype=np.uint8)
    lengths = np.ascontiguousarray(enc["lengths"], dtype=np.int32)
    cdf = np.ascontiguousarray(enc["cdf"], dtype=np.uint16)
    amax = np.ascontiguousarray(enc["amax"], dtype=np.float32)
    kv_out = np.zeros((L, 2, T, C), dtype=np.uint16)
    sym = np.zeros((2, L, T, C), dtype=np.uint8) if want_symbols else None
    nth = nthreads if nthreads > 0 else max_threads()
    _check(lib().orc_decode(_p(data), int(enc["stream_bytes"]), _p(lengths), _p(cdf), _p(amax),
                            L, T, C, chunk_tokens, _p(k), len(k), _p(v), len(v), _p(kv_out),
                            _p(sym) if sym is not None else None, nth), "decode")
    return (kv_out, sym) if want_symbols else kv_out


def encode_tiles(kv_bits: np.ndarray, chunk_tokens: int, kspecs, vspecs, tiles,
                 nthreads: int = 0) -> list:
    """Encode only the listed tiles (index = (group * 2 + kv) * L + layer).
    Returns one dict per tile with amax, cdf, lengths and stream bytes."""
    kv = np.ascontiguousarray(kv_bits, dtype=np.uint16)
    L, _, T = kv.shape[:3]
    C = int(np.prod(kv.shape[3:]))
    k, v = _specs(kspecs), _specs(vspecs)
    kb = layer_bins(L, k)
    vb = layer_bins(L, v)
    gs, gc = groups(T, chunk_tokens)
    tl = np.ascontiguousarray(np.asarray(tiles, dtype=np.int64))
    ns, nc = [], []
    for ti in tl:
        g, kvs, l = int(ti) // (2 * L), (int(ti) // L) % 2, int(ti) % L
        ns.append(int(gc[g]))
        nc.append(C * (int((kb, vb)[kvs][l]) + 1))
    ntok, ncdf = sum(ns), sum(nc)
    amax = np.zeros(max(ntok, 1), dtype=np.float32)
    cdf = np.zeros(max(ncdf, 1), dtype=np.uint16)
    lengths = np.zeros(max(ntok, 1), dtype=np.int32)
    cap = max(ntok, 1) * (2 * C + 2)
    out = np.zeros(cap, dtype=np.uint8)
    tb = np.zeros(max(len(tl), 1), dtype=np.int64)
    nth = nthreads if nthreads > 0 else max_threads()
    _check(lib().orc_encode_tiles(_p(kv), L, T, C, chunk_tokens, _p(k), len(k), _p(v), len(v),
                                  _p(tl), len(tl), _p(amax), _p(cdf), _p(lengths), _p(out), cap,
                                  _p(tb), nth), "encode_tiles")
    res, to, co = [], 0, 0
    bo = 0
    cap_per_tok = 2 * C + 2
    for i, ti in enumerate(tl):
        n, e = ns[i], nc[i]
        res.append({"tile": int(ti), "amax": amax[to:to + n].copy(),
                    "cdf": cdf[co:co + e].copy(), "lengths": lengths[to:to + n].copy(),
                    "bytes": out[bo:bo + int(tb[i])].copy()})
        to += n
        co += e
        bo += n * cap_per_tok
    return res


def container_size(L, T, nspecs_total, cdf_entries_, stream_bytes) -> int:
    return int(lib().orc_container_size(L, T, nspecs_total, cdf_entries_, stream_bytes))


def serialize(enc: dict, L, T, H, D, chunk_tokens, kspecs, vspecs) -> bytes:
    k, v = _specs(kspecs), _specs(vspecs)
    ent = int(enc["cdf"].size)
    sb = int(enc["stream_bytes"])
    size = container_size(L, T, len(k) + len(v), ent, sb)
    out = np.zeros(size, dtype=np.uint8)
    data = np.ascontiguousarray(enc["bytes"], dtype=np.uint8)
    if data.size == 0:
        data = np.zeros(1, dtype=np.uint8)
    _check(lib().orc_serialize(L, T, H, D, chunk_tokens, _p(k), len(k), _p(v), len(v),
                               _p(np.ascontiguousarray(enc["amax"], dtype=np.float32)),
                               _p(np.ascontiguousarray(enc["lengths"], dtype=np.int32)),
                               _p(np.ascontiguousarray(enc["cdf"], dtype=np.uint16)), ent,
                               _p(data), sb, _p(out), size), "serialize")
    return out.tobytes()


# ---------------------------------------------------------- int8 baseline

def int8_quantize_row(x_bits: np.ndarray):
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    q = np.zeros(x.size, dtype=np.int8)
    a = ct.c_float(0.0)
    _check(lib().orc_int8_quantize_row(_p(x), x.size, ct.byref(a), _p(q)), "int8_quantize_row")
    return float(np.float32(a.value)), q


def int8_dequant_row(q: np.ndarray, amax: float) -> np.ndarray:
    q = np.ascontiguousarray(q, dtype=np.int8)
    y = np.zeros(q.size, dtype=np.uint16)
    lib().orc_int8_dequant_row(_p(q), q.size, ct.c_float(amax), _p(y))
    return y


def int8_encode(kv_bits: np.ndarray, nthreads: int = 0):
    """Rows of the last axis: returns (q int8 same shape, scales float32 [rows])."""
    kv = np.ascontiguousarray(kv_bits, dtype=np.uint16)
    C = kv.shape[-1]
    rows = kv.size // C
    q = np.zeros(kv.shape, dtype=np.int8)
    sc = np.zeros(rows, dtype=np.float32)
    _check(lib().orc_int8_encode(_p(kv), rows, C, _p(q), _p(sc),
                                 nthreads if nthreads > 0 else max_threads()), "int8_encode")
    return q, sc


def int8_decode(q: np.ndarray, scales: np.ndarray, nthreads: int = 0) -> np.ndarray:
    q = np.ascontiguousarray(q, dtype=np.int8)
    sc = np.ascontiguousarray(scales, dtype=np.float32)
    C = q.shape[-1]
    out = np.zeros(q.shape, dtype=np.uint16)
    lib().orc_int8_decode(_p(q), _p(sc), q.size // C, C, _p(out),
                          nthreads if nthreads > 0 else max_threads())
    return out
