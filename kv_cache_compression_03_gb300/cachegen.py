"""Python binding of the CacheGen codec's C ABI (include/cachegen.h).

The functions named ``cg_*`` mirror the C entry points one to one and only
marshal arguments: every step of encoding and decoding runs in the CUDA
kernels of ``libcachegen.so``. Device buffers are torch tensors (torch is
used for device memory and streams only). There is no CPU fallback: if the
library is missing or no GPU is present, the calls raise.

``Codec`` wraps a plan with its buffers for the common case; ``preset_specs``
gives the per-layer bin counts of the LMCache presets ("LMCache 中的 KV Cache
压缩：CacheGen 编解码原理、配置方式与源码解析", §1: the first 10 K layers and the
first 2 V layers use 32 bins, the rest 16; fewer than 10 layers: all 32).
"""
from __future__ import annotations

import contextlib
import ctypes as ct
import os
import threading
from dataclasses import dataclass

CG_OK, CG_ERR_INVALID_ARG, CG_ERR_SPEC, CG_ERR_CAPACITY = 0, 1, 2, 3
CG_ERR_NONFINITE, CG_ERR_CORRUPT, CG_ERR_TIMEOUT, CG_ERR_CUDA, CG_ERR_UNSUPPORTED = 4, 5, 6, 7, 8


class cg_quant_spec(ct.Structure):
    _fields_ = [("start_layer", ct.c_int32), ("end_layer", ct.c_int32), ("bins", ct.c_int32)]


class cg_config(ct.Structure):
    _fields_ = [("num_layers", ct.c_int32), ("num_tokens", ct.c_int32),
                ("num_heads", ct.c_int32), ("head_size", ct.c_int32),
                ("chunk_tokens", ct.c_int32),
                ("kspecs", ct.POINTER(cg_quant_spec)), ("n_kspecs", ct.c_int32),
                ("vspecs", ct.POINTER(cg_quant_spec)), ("n_vspecs", ct.c_int32)]


class cg_sizes(ct.Structure):
    _fields_ = [("workspace_bytes", ct.c_size_t), ("max_stream_bytes", ct.c_size_t),
                ("cdf_entries", ct.c_size_t), ("num_streams", ct.c_size_t),
                ("num_scales", ct.c_size_t), ("raw_bytes", ct.c_size_t),
                ("num_groups", ct.c_int32), ("num_tiles", ct.c_int32),
                ("encode_launches", ct.c_int32), ("decode_launches", ct.c_int32),
                ("num_objects", ct.c_int32)]


class cg_encoded(ct.Structure):
    _fields_ = [("bytestream", ct.c_void_p), ("bytestream_capacity", ct.c_size_t),
                ("lengths", ct.c_void_p), ("cdf", ct.c_void_p), ("amax", ct.c_void_p)]


class cg_kernel_profile(ct.Structure):
    _fields_ = [("kernel", ct.c_char_p), ("launches", ct.c_int64), ("total_ms", ct.c_double)]


class CacheGenError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {cg_status_string(status)} ({status})")
        self.status = status


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return os.path.join(os.path.dirname(os.path.abspath(__file__)), "_build", "libcachegen.so")


def load(build_if_missing: bool = True) -> ct.CDLL:
    """Load libcachegen.so (building it with nvcc when absent)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if build_if_missing:
            from . import build as _build
            path = _build.build()
        _lib = _open(path)
        return _lib


@contextlib.contextmanager
def use_library(path: str):
    """Run the calls of this module against another build of the library
    (the tests' variants with forced slow paths), then switch back."""
    global _lib
    L = _open(path)
    with _lock:
        prev, _lib = _lib, L
    try:
        yield L
    finally:
        with _lock:
            _lib = prev


def _open(path: str) -> ct.CDLL:
    if not os.path.exists(path):
        raise ImportError(f"libcachegen.so not found at {path}; run build() first")
    L = ct.CDLL(path)
    P, sz, u64 = ct.c_void_p, ct.c_size_t, ct.c_uint64
    st = ct.c_int
    sigs = {
        "cg_plan_create": (st, [ct.POINTER(cg_config), ct.POINTER(ct.c_void_p)]),
        "cg_plan_destroy": (None, [P]),
        "cg_plan_sizes": (st, [P, ct.POINTER(cg_sizes)]),
        "cg_plan_config": (st, [P, ct.POINTER(cg_config), ct.POINTER(cg_quant_spec),
                                ct.c_int32, ct.POINTER(cg_quant_spec), ct.c_int32]),
        "cg_encode": (st, [P, P, P, sz, ct.POINTER(cg_encoded), P]),
        "cg_decode": (st, [P, ct.POINTER(cg_encoded), u64, P, sz, P, P]),
        "cg_last_device_error": (st, [P, P, ct.POINTER(ct.c_int), ct.POINTER(u64), P]),
        "cg_container_size": (st, [P, u64, ct.POINTER(sz)]),
        "cg_serialize": (st, [P, ct.POINTER(cg_encoded), u64, P, sz, ct.POINTER(sz), P]),
        "cg_container_open": (st, [P, sz, ct.POINTER(ct.c_void_p), ct.POINTER(u64)]),
        "cg_deserialize": (st, [P, P, sz, ct.POINTER(cg_encoded), P]),
        "cg_status_string": (ct.c_char_p, [st]),
        "cg_encode_noalloc": (st, [P, P, ct.POINTER(cg_encoded), P, P]),
        "cg_object_range": (st, [P, ct.c_int32, ct.POINTER(ct.c_int32),
                                 ct.POINTER(ct.c_int32)]),
        "cg_object_streams": (st, [P, P, ct.c_int32, ct.POINTER(u64), ct.POINTER(u64), P]),
        "cg_object_container_size": (st, [P, ct.c_int32, u64, ct.POINTER(sz)]),
        "cg_serialize_object": (st, [P, ct.POINTER(cg_encoded), P, ct.c_int32, P, sz,
                                     ct.POINTER(sz), P]),
        "cg_deserialize_objects": (st, [P, ct.c_int32, ct.POINTER(ct.c_void_p),
                                        ct.POINTER(sz), ct.POINTER(cg_encoded),
                                        ct.POINTER(u64), P]),
        "cg_int8_encode": (st, [P, ct.c_int64, ct.c_int32, P, P, P, P]),
        "cg_int8_decode": (st, [P, P, ct.c_int64, ct.c_int32, P, P]),
        "cg_profile_enable": (st, [P, ct.c_int32]),
        "cg_profile_read": (st, [P, ct.POINTER(cg_kernel_profile), ct.c_int32,
                                 ct.POINTER(ct.c_int32)]),
    }
    for name, (res, args) in sigs.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    return L


def _check(st: int, what: str):
    if st != CG_OK:
        raise CacheGenError(st, what)


def _stream_handle(stream=None):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ct.c_void_p(s.cuda_stream)


def _ptr(t) -> int:
    return t.data_ptr() if t is not None else 0


def _check_status_buffer(status_out, what: str) -> None:
    """The C side copies a 16-byte status block into status_out: it must be
    a CUDA tensor of at least 16 bytes (a smaller one would be overrun)."""
    if status_out is None or not getattr(status_out, "is_cuda", False):
        raise ValueError(f"{what}: status_out must be a CUDA tensor")
    if status_out.numel() * status_out.element_size() < 16:
        raise ValueError(f"{what}: status_out must hold at least 16 bytes")


# ------------------------------------------------------------ C ABI mirror

def cg_status_string(status: int) -> str:
    try:
        return load(build_if_missing=False).cg_status_string(status).decode()
    except Exception:  # library not loadable: still give a message
        return f"status {status}"


def _specs_array(specs):
    arr = (cg_quant_spec * len(specs))()
    for i, (s, e, b) in enumerate(specs):
        arr[i] = cg_quant_spec(int(s), int(e), int(b))
    return arr


def cg_plan_create(num_layers, num_tokens, num_heads, head_size, chunk_tokens, kspecs, vspecs):
    """Validate a configuration and return an opaque plan handle (int)."""
    ka, va = _specs_array(kspecs), _specs_array(vspecs)
    cfg = cg_config(num_layers, num_tokens, num_heads, head_size, chunk_tokens,
                    ka, len(kspecs), va, len(vspecs))
    h = ct.c_void_p()
    _check(load().cg_plan_create(ct.byref(cfg), ct.byref(h)), "cg_plan_create")
    return h.value


def cg_plan_destroy(plan) -> None:
    if plan:
        load().cg_plan_destroy(ct.c_void_p(plan))


def cg_plan_sizes(plan) -> cg_sizes:
    s = cg_sizes()
    _check(load().cg_plan_sizes(ct.c_void_p(plan), ct.byref(s)), "cg_plan_sizes")
    return s


def cg_plan_config(plan):
    """The configuration of a plan: (num_layers, num_tokens, num_heads,
    head_size, chunk_tokens, kspecs, vspecs) with the specs as
    (start_layer, end_layer, bins) triples."""
    lib = load()
    cfg = cg_config()
    st = lib.cg_plan_config(ct.c_void_p(plan), ct.byref(cfg), None, 0, None, 0)
    if st not in (CG_OK, CG_ERR_CAPACITY):
        _check(st, "cg_plan_config")
    ka = (cg_quant_spec * max(cfg.n_kspecs, 1))()
    va = (cg_quant_spec * max(cfg.n_vspecs, 1))()
    _check(lib.cg_plan_config(ct.c_void_p(plan), ct.byref(cfg), ka, cfg.n_kspecs, va,
                              cfg.n_vspecs), "cg_plan_config")
    ks = [(ka[i].start_layer, ka[i].end_layer, ka[i].bins) for i in range(cfg.n_kspecs)]
    vs = [(va[i].start_layer, va[i].end_layer, va[i].bins) for i in range(cfg.n_vspecs)]
    return (cfg.num_layers, cfg.num_tokens, cfg.num_heads, cfg.head_size, cfg.chunk_tokens,
            ks, vs)


def _encoded_struct(bytestream, lengths, cdf, amax) -> cg_encoded:
    return cg_encoded(_ptr(bytestream), bytestream.numel() * bytestream.element_size(),
                      _ptr(lengths), _ptr(cdf), _ptr(amax))


def cg_encode(plan, kv, workspace, bytestream, lengths, cdf, amax, stream=None) -> None:
    enc = _encoded_struct(bytestream, lengths, cdf, amax)
    _check(load().cg_encode(ct.c_void_p(plan), ct.c_void_p(_ptr(kv)), ct.c_void_p(_ptr(workspace)),
                            workspace.numel(), ct.byref(enc), _stream_handle(stream)), "cg_encode")


def cg_encode_noalloc(plan, kv, bytestream, lengths, cdf, amax, status_out, stream=None) -> None:
    """cg_encode with the library's fixed scratch array instead of a
    workspace, for callers that cannot allocate device memory at encode time
    (see include/cachegen.h). status_out: a device tensor of >= 16 bytes that
    receives the status word and total stream bytes; read it with
    cg_last_device_error(plan, status_out)."""
    _check_status_buffer(status_out, "cg_encode_noalloc")
    enc = _encoded_struct(bytestream, lengths, cdf, amax)
    _check(load().cg_encode_noalloc(ct.c_void_p(plan), ct.c_void_p(_ptr(kv)), ct.byref(enc),
                                    ct.c_void_p(_ptr(status_out)), _stream_handle(stream)),
           "cg_encode_noalloc")


def cg_decode(plan, bytestream, lengths, cdf, amax, stream_bytes, workspace, kv_out,
              stream=None) -> None:
    enc = _encoded_struct(bytestream, lengths, cdf, amax)
    _check(load().cg_decode(ct.c_void_p(plan), ct.byref(enc), int(stream_bytes),
                            ct.c_void_p(_ptr(workspace)), workspace.numel(),
                            ct.c_void_p(_ptr(kv_out)), _stream_handle(stream)), "cg_decode")


def cg_int8_encode(kv, rows, channels, q_out, scales_out, status_out, stream=None) -> None:
    """Int8 baseline encode (include/cachegen.h): kv bf16 [rows][channels]
    into q_out int8 [rows][channels] and scales_out fp32 [rows]; status_out
    (>= 16 bytes) gets the device status, read with
    cg_last_device_error(None, status_out)."""
    _check_status_buffer(status_out, "cg_int8_encode")
    _check(load().cg_int8_encode(ct.c_void_p(_ptr(kv)), int(rows), int(channels),
                                 ct.c_void_p(_ptr(q_out)), ct.c_void_p(_ptr(scales_out)),
                                 ct.c_void_p(_ptr(status_out)), _stream_handle(stream)),
           "cg_int8_encode")


def cg_int8_decode(q, scales, rows, channels, kv_out, stream=None) -> None:
    """Int8 baseline decode: q int8 [rows][channels] and scales fp32 [rows]
    into kv_out bf16 [rows][channels]."""
    _check(load().cg_int8_decode(ct.c_void_p(_ptr(q)), ct.c_void_p(_ptr(scales)), int(rows),
                                 int(channels), ct.c_void_p(_ptr(kv_out)), _stream_handle(stream)),
           "cg_int8_decode")


def cg_object_range(plan, obj):
    """(first token, token count) of an object of the plan."""
    t0, n = ct.c_int32(0), ct.c_int32(0)
    _check(load().cg_object_range(ct.c_void_p(plan), int(obj), ct.byref(t0), ct.byref(n)),
           "cg_object_range")
    return t0.value, n.value


def cg_object_streams(plan, workspace, obj, stream=None):
    """(offset, bytes) of an object's streams in the last encoded bytestream."""
    off, nb = ct.c_uint64(0), ct.c_uint64(0)
    _check(load().cg_object_streams(ct.c_void_p(plan), ct.c_void_p(_ptr(workspace)), int(obj),
                                    ct.byref(off), ct.byref(nb), _stream_handle(stream)),
           "cg_object_streams")
    return off.value, nb.value


def cg_object_container_size(plan, obj, stream_bytes) -> int:
    n = ct.c_size_t(0)
    _check(load().cg_object_container_size(ct.c_void_p(plan), int(obj), int(stream_bytes),
                                           ct.byref(n)), "cg_object_container_size")
    return n.value


def cg_serialize_object(plan, bytestream, lengths, cdf, amax, workspace, obj, host_out,
                        stream=None) -> int:
    enc = _encoded_struct(bytestream, lengths, cdf, amax)
    w = ct.c_size_t(0)
    _check(load().cg_serialize_object(ct.c_void_p(plan), ct.byref(enc),
                                      ct.c_void_p(_ptr(workspace)), int(obj),
                                      ct.c_void_p(host_out.data_ptr()), host_out.numel(),
                                      ct.byref(w), _stream_handle(stream)), "cg_serialize_object")
    return w.value


def cg_deserialize_objects(plan, hosts, bytestream, lengths, cdf, amax, stream=None) -> int:
    """hosts: uint8 CPU tensors, one container per object in object order.
    Returns the total stream bytes."""
    n = len(hosts)
    ptrs = (ct.c_void_p * max(n, 1))(*[h.data_ptr() for h in hosts])
    lens = (ct.c_size_t * max(n, 1))(*[h.numel() for h in hosts])
    enc = _encoded_struct(bytestream, lengths, cdf, amax)
    sb = ct.c_uint64(0)
    _check(load().cg_deserialize_objects(ct.c_void_p(plan), n, ptrs, lens, ct.byref(enc),
                                         ct.byref(sb), _stream_handle(stream)),
           "cg_deserialize_objects")
    return sb.value


def int8_encode(kv, stream=None, sync: bool = True):
    """Int8 baseline encode of a contiguous bf16 cuda tensor whose last
    dimension is the row (a KV cache [L, 2, T, H, D] is taken as rows of
    H*D). Returns (q int8 of kv's shape, scales fp32 [rows], status tensor);
    with sync, a device error is raised."""
    import torch
    assert kv.dtype == torch.bfloat16 and kv.is_cuda and kv.is_contiguous()
    C = kv.shape[-1] if kv.dim() != 5 else kv.shape[-2] * kv.shape[-1]
    rows = kv.numel() // C if C else 0
    q = torch.empty(kv.shape, dtype=torch.int8, device=kv.device)
    scales = torch.empty(rows, dtype=torch.float32, device=kv.device)
    status = torch.empty(16, dtype=torch.uint8, device=kv.device)
    cg_int8_encode(kv, rows, C, q, scales, status, stream)
    if sync:
        st, _ = cg_last_device_error(None, status, stream)
        _check(st, "cg_int8_encode (device)")
    return q, scales, status


def int8_decode(q, scales, stream=None):
    """Int8 baseline decode: the bf16 tensor of q's shape."""
    import torch
    C = q.shape[-1] if q.dim() != 5 else q.shape[-2] * q.shape[-1]
    rows = q.numel() // C if C else 0
    out = torch.empty(q.shape, dtype=torch.bfloat16, device=q.device)
    cg_int8_decode(q, scales, rows, C, out, stream)
    return out


def cg_last_device_error(plan, workspace, stream=None):
    """Wait for the stream; return (device status, total stream bytes)."""
    st = ct.c_int(0)
    tot = ct.c_uint64(0)
    _check(load().cg_last_device_error(ct.c_void_p(plan or 0), ct.c_void_p(_ptr(workspace)),
                                       ct.byref(st), ct.byref(tot), _stream_handle(stream)),
           "cg_last_device_error")
    return st.value, tot.value


def cg_container_size(plan, stream_bytes) -> int:
    n = ct.c_size_t(0)
    _check(load().cg_container_size(ct.c_void_p(plan), int(stream_bytes), ct.byref(n)),
           "cg_container_size")
    return n.value


def cg_serialize(plan, bytestream, lengths, cdf, amax, stream_bytes, host_out, stream=None) -> int:
    """Write the container into host_out (a uint8 CPU tensor, ideally
    pinned); returns the bytes written."""
    enc = _encoded_struct(bytestream, lengths, cdf, amax)
    n = ct.c_size_t(0)
    _check(load().cg_serialize(ct.c_void_p(plan), ct.byref(enc), int(stream_bytes),
                               ct.c_void_p(host_out.data_ptr()), host_out.numel(), ct.byref(n),
                               _stream_handle(stream)), "cg_serialize")
    return n.value


def cg_container_open(host_in):
    """Parse a container header (uint8 CPU tensor); return (plan, stream_bytes)."""
    h = ct.c_void_p()
    sb = ct.c_uint64(0)
    _check(load().cg_container_open(ct.c_void_p(host_in.data_ptr()), host_in.numel(),
                                    ct.byref(h), ct.byref(sb)), "cg_container_open")
    return h.value, sb.value


def cg_deserialize(plan, host_in, bytestream, lengths, cdf, amax, stream=None) -> None:
    enc = _encoded_struct(bytestream, lengths, cdf, amax)
    _check(load().cg_deserialize(ct.c_void_p(plan), ct.c_void_p(host_in.data_ptr()),
                                 host_in.numel(), ct.byref(enc), _stream_handle(stream)),
           "cg_deserialize")


def cg_profile_enable(plan, max_launches: int) -> None:
    _check(load().cg_profile_enable(ct.c_void_p(plan), int(max_launches)), "cg_profile_enable")


def cg_profile_read(plan) -> dict:
    """{kernel name: (launches, total ms)} since the last read."""
    arr = (cg_kernel_profile * 16)()
    n = ct.c_int32(0)
    _check(load().cg_profile_read(ct.c_void_p(plan), arr, 16, ct.byref(n)), "cg_profile_read")
    return {arr[i].kernel.decode(): (int(arr[i].launches), float(arr[i].total_ms))
            for i in range(min(n.value, 16))}


# ------------------------------------------------------------- convenience

def preset_specs(num_layers: int):
    """(kspecs, vspecs) of the LMCache presets for a model with num_layers
    layers: K's first 10 and V's first 2 layers at 32 bins, the rest at 16;
    with fewer than 10 layers every layer uses 32 bins."""
    L = int(num_layers)
    if L <= 0:
        raise ValueError("num_layers must be positive")
    if L < 10:
        return [(0, L, 32)], [(0, L, 32)]
    k = [(0, 10, 32)] + ([(10, L, 16)] if L > 10 else [])
    v = [(0, 2, 32), (2, L, 16)]
    return k, v


@dataclass
class Encoded:
    """Device buffers of one encoded KV blob."""
    bytestream: "object"   # uint8 [capacity]
    lengths: "object"      # int32 [2*L*T]
    cdf: "object"          # uint16 (stored as int16) [cdf_entries]
    amax: "object"         # float32 [2, L, T]
    stream_bytes: int

    def nbytes(self) -> int:
        return int(self.stream_bytes) + self.lengths.numel() * 4 + self.cdf.numel() * 2 + \
            self.amax.numel() * 4


class Codec:
    """A plan plus its device buffers, for encoding/decoding one shape."""

    def __init__(self, num_layers, num_tokens, num_heads, head_size, chunk_tokens=256,
                 kspecs=None, vspecs=None, device="cuda"):
        import torch
        if kspecs is None or vspecs is None:
            k, v = preset_specs(num_layers)
            kspecs = kspecs or k
            vspecs = vspecs or v
        self.L, self.T, self.H, self.D = num_layers, num_tokens, num_heads, head_size
        self.chunk_tokens = chunk_tokens
        self.kspecs, self.vspecs = list(kspecs), list(vspecs)
        self.plan = cg_plan_create(num_layers, num_tokens, num_heads, head_size, chunk_tokens,
                                   self.kspecs, self.vspecs)
        self.sizes = cg_plan_sizes(self.plan)
        self.device = torch.device(device)
        self.workspace = torch.empty(self.sizes.workspace_bytes, dtype=torch.uint8,
                                     device=self.device)

    def __del__(self):
        try:
            cg_plan_destroy(self.plan)
        except Exception:
            pass

    def alloc_encoded(self, capacity=None) -> Encoded:
        import torch
        cap = int(capacity or self.sizes.max_stream_bytes)
        cap = (cap + 15) // 16 * 16
        d = self.device
        return Encoded(torch.empty(cap, dtype=torch.uint8, device=d),
                       torch.empty(self.sizes.num_streams, dtype=torch.int32, device=d),
                       torch.empty(self.sizes.cdf_entries, dtype=torch.int16, device=d),
                       torch.empty((2, self.L, self.T), dtype=torch.float32, device=d), 0)

    def encode(self, kv, out: Encoded | None = None, sync: bool = True, stream=None) -> Encoded:
        """kv: bf16 cuda tensor [L, 2, T, H, D] (contiguous)."""
        import torch
        assert kv.dtype == torch.bfloat16 and kv.is_cuda and kv.is_contiguous()
        assert kv.numel() == self.sizes.raw_bytes // 2
        out = out or self.alloc_encoded()
        cg_encode(self.plan, kv, self.workspace, out.bytestream, out.lengths, out.cdf, out.amax,
                  stream)
        if sync:
            st, total = cg_last_device_error(self.plan, self.workspace, stream)
            _check(st, "cg_encode (device)")
            out.stream_bytes = total
        return out

    def decode(self, enc: Encoded, kv_out=None, sync: bool = True, stream=None):
        import torch
        if kv_out is None:
            kv_out = torch.empty((self.L, 2, self.T, self.H, self.D), dtype=torch.bfloat16,
                                 device=self.device)
        cg_decode(self.plan, enc.bytestream, enc.lengths, enc.cdf, enc.amax, enc.stream_bytes,
                  self.workspace, kv_out, stream)
        if sync:
            st, _ = cg_last_device_error(self.plan, self.workspace, stream)
            _check(st, "cg_decode (device)")
        return kv_out

    def to_bytes(self, enc: Encoded, host_out=None, stream=None):
        """Serialise to a uint8 CPU tensor (pinned unless host_out is given)."""
        import torch
        n = cg_container_size(self.plan, enc.stream_bytes)
        if host_out is None:
            host_out = torch.empty(n, dtype=torch.uint8, pin_memory=True)
        w = cg_serialize(self.plan, enc.bytestream, enc.lengths, enc.cdf, enc.amax,
                         enc.stream_bytes, host_out, stream)
        return host_out[:w]

    def object_bytes(self, enc: Encoded, stream=None):
        """One container per object (uint8 CPU tensors) of the blob that the
        last encode with this codec wrote into enc."""
        import torch
        out = []
        for o in range(self.sizes.num_objects):
            _, nb = cg_object_streams(self.plan, self.workspace, o, stream)
            host = torch.empty(cg_object_container_size(self.plan, o, nb), dtype=torch.uint8,
                               pin_memory=True)
            w = cg_serialize_object(self.plan, enc.bytestream, enc.lengths, enc.cdf, enc.amax,
                                    self.workspace, o, host, stream)
            out.append(host[:w])
        return out

    def from_object_bytes(self, hosts, out: Encoded | None = None, stream=None) -> Encoded:
        """Put the containers of all objects back for one decode."""
        out = out or self.alloc_encoded()
        out.stream_bytes = cg_deserialize_objects(self.plan, hosts, out.bytestream, out.lengths,
                                                  out.cdf, out.amax, stream)
        return out

    @staticmethod
    def from_bytes(host_in, device="cuda", stream=None):
        """Open a container (uint8 CPU tensor); return (codec, encoded)."""
        plan, sb = cg_container_open(host_in)
        try:
            L, T, H, D, ch, kspecs, vspecs = cg_plan_config(plan)
        finally:
            cg_plan_destroy(plan)
        codec = Codec(L, T, H, D, ch, kspecs, vspecs, device=device)
        enc = codec.alloc_encoded(capacity=max(16, sb))
        enc.stream_bytes = sb
        cg_deserialize(codec.plan, host_in, enc.bytestream, enc.lengths, enc.cdf, enc.amax,
                       stream)
        return codec, enc
