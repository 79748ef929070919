"""Host-side checks of the C ABI (no GPU needed): the library builds and
exports every function include/cachegen.h declares, configuration
validation matches the oracle's, sizes follow the layout, and a container
written by the oracle opens with the same plan."""
import ctypes as ct
import struct
import os
import re
import subprocess

import numpy as np
import pytest

from kv_cache_compression_03_gb300 import cachegen as cg
from kv_cache_compression_03_gb300 import synthetic

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "cachegen.h")


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(cg_[a-z_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    return cg.load()


def test_header_declares_boundary():
    names = _declared()
    for want in ("cg_plan_create", "cg_plan_destroy", "cg_plan_sizes", "cg_encode", "cg_decode",
                 "cg_last_device_error", "cg_container_size", "cg_serialize",
                 "cg_container_open", "cg_deserialize", "cg_status_string"):
        assert want in names


def test_library_exports_every_declared_symbol(lib):
    path = cg.library_path()
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r" T (\w+)$", out, flags=re.M))
    for name in _declared():
        assert name in exported, name
        assert getattr(lib, name) is not None


def test_header_compiles_as_c():
    r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-fsyntax-only", "-x", "c",
                        HEADER], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def _plan(L=32, T=1024, H=8, D=128, ch=256, k=None, v=None):
    if k is None:
        k, v = cg.preset_specs(L)
    return cg.cg_plan_create(L, T, H, D, ch, k, v)


def test_plan_sizes_match_layout(orc):
    for name in synthetic.WORKLOADS:
        p = synthetic.WORKLOADS[name]
        k, v = synthetic.workload_specs(name)
        for ch in p["chunk_tokens"]:
            plan = cg.cg_plan_create(p["L"], p["T"], p["H"], p["D"], ch, k, v)
            try:
                s = cg.cg_plan_sizes(plan)
                C = p["H"] * p["D"]
                assert s.num_streams == 2 * p["L"] * p["T"] == s.num_scales
                assert s.raw_bytes == 2 * p["L"] * p["T"] * C * 2
                assert s.num_groups == len(orc.groups(p["T"], ch)[0])
                assert s.num_tiles == s.num_groups * 2 * p["L"]
                assert s.cdf_entries == orc.cdf_entries(p["L"], p["T"], C, ch, k, v)
                assert s.max_stream_bytes >= s.num_streams * (C + 1)
                assert s.encode_launches >= 1 and s.decode_launches >= 1
                assert s.workspace_bytes > 0
            finally:
                cg.cg_plan_destroy(plan)


@pytest.mark.parametrize("k,v", [
    ([(0, 10, 32), (9, 32, 16)], [(0, 32, 16)]),
    ([(0, 32, 16)], [(0, 2, 32), (3, 32, 16)]),
    ([(0, 32, 15)], [(0, 32, 16)]),
    ([(0, 32, 2)], [(0, 32, 16)]),
    ([(0, 32, 66)], [(0, 32, 16)]),
    ([(0, 33, 16)], [(0, 32, 16)]),
])
def test_plan_rejects_bad_specs(orc, k, v):
    with pytest.raises(cg.CacheGenError) as e:
        _plan(k=k, v=v)
    assert e.value.status == cg.CG_ERR_SPEC
    # the oracle rejects the same lists
    with pytest.raises(orc.OracleError):
        orc.layer_bins(32, k)
        orc.layer_bins(32, v)


@pytest.mark.parametrize("args,code", [
    ((0, 1024, 8, 128, 256), cg.CG_ERR_INVALID_ARG),
    ((32, 0, 8, 128, 256), cg.CG_ERR_INVALID_ARG),
    ((32, 1024, 8, 128, 0), cg.CG_ERR_INVALID_ARG),
    ((32, 1024, 1, 12, 256), cg.CG_ERR_INVALID_ARG),     # C not a multiple of 8
    ((32, 1024, 64, 128, 256), cg.CG_ERR_UNSUPPORTED),   # C = 8192 > 4096
    ((300, 16, 8, 128, 256), cg.CG_ERR_UNSUPPORTED),     # more than 256 layers
])
def test_plan_rejects_bad_shapes(args, code):
    L = args[0]
    k, v = cg.preset_specs(max(L, 1))
    with pytest.raises(cg.CacheGenError) as e:
        cg.cg_plan_create(*args, k, v)
    assert e.value.status == code


def test_large_tables_are_planned_in_channel_parts():
    """CDF tables beyond shared memory (C = 4096 at 32 and 64 bins) are coded
    and decoded in channel parts, so every shape up to 4096 channels plans."""
    for bins in (16, 32, 64):
        plan = cg.cg_plan_create(2, 16, 32, 128, 256, [(0, 2, bins)], [(0, 2, bins)])
        try:
            assert cg.cg_plan_sizes(plan).workspace_bytes > 0
        finally:
            cg.cg_plan_destroy(plan)


def test_preset_specs():
    assert cg.preset_specs(32) == ([(0, 10, 32), (10, 32, 16)], [(0, 2, 32), (2, 32, 16)])
    assert cg.preset_specs(40) == ([(0, 10, 32), (10, 40, 16)], [(0, 2, 32), (2, 40, 16)])
    assert cg.preset_specs(6) == ([(0, 6, 32)], [(0, 6, 32)])
    assert cg.preset_specs(10) == ([(0, 10, 32)], [(0, 2, 32), (2, 10, 16)])
    for L in (12, 32, 40):
        assert cg.preset_specs(L) == synthetic.workload_specs(
            {12: "opt125m_t256", 32: "mistral7b_t1k", 40: "glm4_9b_t32k"}[L])


def test_container_open_reads_oracle_container(orc):
    import torch
    name = "opt125m_t256"
    kv = synthetic.generate(name, num_tokens=300)
    L, _, T, C = kv.shape
    k, v = synthetic.workload_specs(name)
    enc = orc.encode(kv, 256, k, v)
    blob = orc.serialize(enc, L, T, 12, 64, 256, k, v)
    host = torch.from_numpy(np.frombuffer(blob, dtype=np.uint8).copy())
    plan, sb = cg.cg_container_open(host)
    try:
        assert sb == enc["stream_bytes"]
        assert cg.cg_container_size(plan, sb) == len(blob)
        s = cg.cg_plan_sizes(plan)
        assert s.cdf_entries == enc["cdf"].size and s.num_streams == 2 * L * T
    finally:
        cg.cg_plan_destroy(plan)
    # a damaged header is rejected
    bad = host.clone()
    bad[0] = 0
    with pytest.raises(cg.CacheGenError) as e:
        cg.cg_container_open(bad)
    assert e.value.status == cg.CG_ERR_CORRUPT
    short = host[:-1].clone()
    with pytest.raises(cg.CacheGenError) as e:
        cg.cg_container_open(short)
    assert e.value.status == cg.CG_ERR_CORRUPT


def test_status_strings(lib):
    assert cg.cg_status_string(0) == "ok"
    assert "capacity" in cg.cg_status_string(cg.CG_ERR_CAPACITY)


def test_int8_argument_checks(lib):
    """Argument errors of the int8 baseline calls come back before any
    device work is enqueued."""
    P = ct.c_void_p
    fake = P(4096)  # never dereferenced: every call below fails validation
    assert lib.cg_int8_encode(fake, 4, 12, fake, fake, fake, None) == cg.CG_ERR_INVALID_ARG
    assert lib.cg_int8_encode(fake, -1, 16, fake, fake, fake, None) == cg.CG_ERR_INVALID_ARG
    assert lib.cg_int8_encode(fake, 4, 4104, fake, fake, fake, None) == cg.CG_ERR_UNSUPPORTED
    assert lib.cg_int8_encode(fake, 4, 16, fake, fake, None, None) == cg.CG_ERR_INVALID_ARG
    assert lib.cg_int8_encode(P(4098), 4, 16, fake, fake, fake, None) == cg.CG_ERR_INVALID_ARG
    assert lib.cg_int8_encode(fake, 4, 16, P(4097), fake, fake, None) == cg.CG_ERR_INVALID_ARG
    assert lib.cg_int8_encode(None, 4, 16, fake, fake, fake, None) == cg.CG_ERR_INVALID_ARG
    assert lib.cg_int8_decode(fake, fake, 4, 0, fake, None) == cg.CG_ERR_INVALID_ARG
    assert lib.cg_int8_decode(fake, fake, 4, 8192, fake, None) == cg.CG_ERR_UNSUPPORTED
    assert lib.cg_int8_decode(fake, fake, 4, 16, P(4104), None) == cg.CG_ERR_INVALID_ARG
    assert lib.cg_int8_decode(None, fake, 4, 16, fake, None) == cg.CG_ERR_INVALID_ARG
    assert lib.cg_int8_decode(None, None, 0, 16, None, None) == cg.CG_OK


def _object_containers(orc, name, T, ch):
    p = synthetic.WORKLOADS[name]
    kv = synthetic.generate(name, num_tokens=T)
    k, v = synthetic.workload_specs(name)
    L, C = kv.shape[0], kv.shape[-1]
    blobs = []
    for t0 in range(0, T, ch):
        part = np.ascontiguousarray(kv[:, :, t0:t0 + ch])
        enc = orc.encode(part, ch, k, v)
        blobs.append(orc.serialize(enc, L, part.shape[2], p["H"], p["D"], ch, k, v))
    return p, k, v, L, blobs


def test_object_ranges_and_sizes(orc):
    import torch
    name = "opt125m_t256"
    T, ch = 600, 128
    p, k, v, L, blobs = _object_containers(orc, name, T, ch)
    plan = cg.cg_plan_create(L, T, p["H"], p["D"], ch, k, v)
    try:
        s = cg.cg_plan_sizes(plan)
        assert s.num_objects == 5 == len(blobs)
        for o, blob in enumerate(blobs):
            t0, n = cg.cg_object_range(plan, o)
            assert (t0, n) == (o * ch, min(ch, T - o * ch))
            # the size rule agrees with the oracle's container of the slice
            sb = struct.unpack_from("<Q", blob, 40)[0]
            assert cg.cg_object_container_size(plan, o, sb) == len(blob)
            # and the slice's own plan opens it
            oplan, osb = cg.cg_container_open(torch.from_numpy(np.frombuffer(blob, np.uint8).copy()))
            cg.cg_plan_destroy(oplan)
            assert osb == sb
        for bad in (-1, 5):
            with pytest.raises(cg.CacheGenError):
                cg.cg_object_range(plan, bad)
    finally:
        cg.cg_plan_destroy(plan)


def test_deserialize_objects_checks_headers_first(orc, lib):
    """Containers that are not object i of the plan are rejected before any
    copy (no device is touched here)."""
    import torch
    name = "opt125m_t256"
    T, ch = 600, 256
    p, k, v, L, blobs = _object_containers(orc, name, T, ch)
    plan = cg.cg_plan_create(L, T, p["H"], p["D"], ch, k, v)
    fake = torch.zeros(64, dtype=torch.uint8)  # never written: validation fails first
    hosts = [torch.from_numpy(np.frombuffer(b, np.uint8).copy()) for b in blobs]
    try:
        def call(hs, pl=plan):
            # the C call itself, on the default stream (the binding would ask
            # torch for the current CUDA stream)
            n = len(hs)
            ptrs = (ct.c_void_p * n)(*[h.data_ptr() for h in hs])
            lens = (ct.c_size_t * n)(*[h.numel() for h in hs])
            enc = cg.cg_encoded(fake.data_ptr(), 64, fake.data_ptr(), fake.data_ptr(),
                                fake.data_ptr())
            sb = ct.c_uint64(0)
            st = lib.cg_deserialize_objects(ct.c_void_p(pl), n, ptrs, lens, ct.byref(enc),
                                            ct.byref(sb), None)
            if st != cg.CG_OK:
                raise cg.CacheGenError(st, "cg_deserialize_objects")
        with pytest.raises(cg.CacheGenError) as e:
            call(hosts[:2])                                  # wrong object count
        assert e.value.status == cg.CG_ERR_INVALID_ARG
        with pytest.raises(cg.CacheGenError) as e:
            call([hosts[2], hosts[1], hosts[0]])             # the short tail first
        assert e.value.status == cg.CG_ERR_CORRUPT
        with pytest.raises(cg.CacheGenError) as e:
            call([hosts[0], hosts[1], hosts[2][:-1]])        # truncated
        assert e.value.status == cg.CG_ERR_CORRUPT
        bad = hosts[1].clone()
        bad[12] += 1                                         # token count
        with pytest.raises(cg.CacheGenError) as e:
            call([hosts[0], bad, hosts[2]])
        assert e.value.status == cg.CG_ERR_CORRUPT
        plan2 = cg.cg_plan_create(L, T, p["H"], p["D"], ch, [(0, 12, 16)], v)  # other specs
        try:
            with pytest.raises(cg.CacheGenError) as e:
                call(hosts, plan2)
            assert e.value.status == cg.CG_ERR_CORRUPT
        finally:
            cg.cg_plan_destroy(plan2)
    finally:
        cg.cg_plan_destroy(plan)


def test_plan_config_reports_the_configuration(orc):
    """cg_plan_config gives back the shape and spec lists of a plan, also of
    one opened from a container (from_bytes must recover them)."""
    import torch
    k = [(0, 3, 32), (3, 12, 16)]
    v = [(0, 2, 32), (2, 5, 8), (5, 12, 16)]
    plan = cg.cg_plan_create(12, 700, 12, 64, 128, k, v)
    try:
        assert cg.cg_plan_config(plan) == (12, 700, 12, 64, 128, k, v)
        cfg = cg.cg_config()
        ka = (cg.cg_quant_spec * 2)()
        va = (cg.cg_quant_spec * 2)()   # one short: nothing is copied
        lib = cg.load()
        st = lib.cg_plan_config(ct.c_void_p(plan), ct.byref(cfg), ka, 2, va, 2)
        assert st == cg.CG_ERR_CAPACITY
        assert (cfg.n_kspecs, cfg.n_vspecs, cfg.num_tokens) == (2, 3, 700)
        assert (va[0].start_layer, va[0].end_layer, va[0].bins) == (0, 0, 0)
        assert lib.cg_plan_config(None, ct.byref(cfg), None, 0, None, 0) == cg.CG_ERR_INVALID_ARG
        assert lib.cg_plan_config(ct.c_void_p(plan), ct.byref(cfg), None, 2, None, 0) == \
            cg.CG_ERR_INVALID_ARG
    finally:
        cg.cg_plan_destroy(plan)
    name = "glm4_9b_t32k"
    kv = synthetic.generate(name, num_tokens=260)
    L, _, T, C = kv.shape
    ks, vs = synthetic.workload_specs(name)
    enc = orc.encode(kv, 256, ks, vs)
    blob = orc.serialize(enc, L, T, 2, 128, 256, ks, vs)
    host = torch.from_numpy(np.frombuffer(blob, dtype=np.uint8).copy())
    plan, _ = cg.cg_container_open(host)
    try:
        assert cg.cg_plan_config(plan) == (L, T, 2, 128, 256, [tuple(s) for s in ks],
                                           [tuple(s) for s in vs])
    finally:
        cg.cg_plan_destroy(plan)


def test_encode_decode_argument_checks(lib):
    """cg_encode / cg_decode reject null and misaligned pointers and short
    buffers before anything is enqueued (the fake addresses below are never
    dereferenced: each call fails validation on the host)."""
    plan = _plan(L=2, T=300, H=2, D=64, ch=256, k=[(0, 2, 16)], v=[(0, 2, 32)])
    try:
        s = cg.cg_plan_sizes(plan)
        P = ct.c_void_p
        base = 1 << 20   # 256-byte aligned fake address
        ws = P(base)

        def enc(bs=base, ln=base, cdf=base, am=base, cap=1 << 20):
            return cg.cg_encoded(bs, cap, ln, cdf, am)

        good = enc()
        E = lambda kv, w, wb, e: lib.cg_encode(P(plan), kv, w, wb, ct.byref(e), None)  # noqa: E731
        assert E(None, ws, s.workspace_bytes, good) == cg.CG_ERR_INVALID_ARG
        assert E(P(base), None, s.workspace_bytes, good) == cg.CG_ERR_INVALID_ARG
        assert lib.cg_encode(None, P(base), ws, s.workspace_bytes, ct.byref(good), None) == \
            cg.CG_ERR_INVALID_ARG
        assert lib.cg_encode(P(plan), P(base), ws, s.workspace_bytes, None, None) == \
            cg.CG_ERR_INVALID_ARG
        for bad in (enc(bs=0), enc(ln=0), enc(cdf=0), enc(am=0)):
            assert E(P(base), ws, s.workspace_bytes, bad) == cg.CG_ERR_INVALID_ARG
        assert E(P(base + 8), ws, s.workspace_bytes, good) == cg.CG_ERR_INVALID_ARG   # kv
        assert E(P(base), P(base + 16), s.workspace_bytes, good) == cg.CG_ERR_INVALID_ARG
        for bad in (enc(bs=base + 4), enc(cdf=base + 8), enc(ln=base + 2), enc(am=base + 1)):
            assert E(P(base), ws, s.workspace_bytes, bad) == cg.CG_ERR_INVALID_ARG
        assert E(P(base), ws, s.workspace_bytes - 1, good) == cg.CG_ERR_CAPACITY

        n = s.num_streams
        D = lambda e, sb, w, wb, out: lib.cg_decode(P(plan), ct.byref(e), sb, w, wb, out,  # noqa: E731
                                                    None)
        assert D(good, n, None, s.workspace_bytes, P(base)) == cg.CG_ERR_INVALID_ARG
        assert D(good, n, ws, s.workspace_bytes, None) == cg.CG_ERR_INVALID_ARG
        assert lib.cg_decode(P(plan), None, n, ws, s.workspace_bytes, P(base), None) == \
            cg.CG_ERR_INVALID_ARG
        for bad in (enc(bs=0), enc(ln=0), enc(cdf=0), enc(am=0), enc(bs=base + 4),
                    enc(cdf=base + 2), enc(ln=base + 2), enc(am=base + 2)):
            assert D(bad, n, ws, s.workspace_bytes, P(base)) == cg.CG_ERR_INVALID_ARG
        assert D(good, n, ws, s.workspace_bytes, P(base + 8)) == cg.CG_ERR_INVALID_ARG
        assert D(good, n, P(base + 128), s.workspace_bytes, P(base)) == cg.CG_ERR_INVALID_ARG
        assert D(good, n - 1, ws, s.workspace_bytes, P(base)) == cg.CG_ERR_CORRUPT
        assert D(enc(cap=n), n + 1, ws, s.workspace_bytes, P(base)) == cg.CG_ERR_CAPACITY
        assert D(good, n, ws, 255, P(base)) == cg.CG_ERR_CAPACITY
    finally:
        cg.cg_plan_destroy(plan)


def test_status_buffers_are_checked_before_the_call():
    """The Python binding refuses a status buffer the C side would overrun
    (the C side copies 16 bytes into it)."""
    import torch
    small = torch.zeros(8, dtype=torch.uint8)
    with pytest.raises(ValueError):
        cg.cg_encode_noalloc(0, small, small, small, small, small, small)
    with pytest.raises(ValueError):
        cg.cg_int8_encode(small, 1, 8, small, small, small)
    with pytest.raises(ValueError):
        cg.cg_int8_encode(small, 1, 8, small, small, None)


def _count_layout(C, bins):
    """The encoder's counting layout rule, restated: (channels per thread,
    row groups)."""
    if C >= 1024:
        return 4, 1
    table = C * (bins + 1) * 2
    for w in (4, 2):
        u = C // w
        if C % w == 0 and u <= 256 and 256 % u == 0 and 256 // u <= 8 and \
                (256 // u) * table <= 36 * 1024:
            return w, 256 // u
    return (2 if C >= 512 else 1), 1


@pytest.mark.parametrize("L,T,H,D,k,v", [
    (32, 1024, 8, 128, None, None),                      # 16-bin pairs as 4-bit codes
    (40, 700, 2, 128, [(0, 10, 32), (10, 40, 16)], [(0, 2, 32), (2, 40, 16)]),  # C = 256
    (12, 300, 12, 64, None, None),                       # C = 768: bytes only
    (4, 100, 3, 344, [(0, 4, 16)], [(0, 4, 16)]),        # C = 1032: not a multiple of 32
    (3, 77, 1, 64, [(0, 3, 16)], [(0, 3, 8)]),           # C = 64: row groups of 2 channels
])
def test_workspace_layout(L, T, H, D, k, v):
    """The workspace is the status block, per-tile totals and bases, the
    symbol scratch (one region of T rows per K/V layer pair; 16-bin pairs keep
    4-bit codes when the encoder counts four channels per thread and C is a
    multiple of 32) and one slot of C + 32 bytes per stream."""
    if k is None:
        k, v = cg.preset_specs(L)
    C = H * D
    plan = cg.cg_plan_create(L, T, H, D, 256, k, v)
    try:
        s = cg.cg_plan_sizes(plan)
        up = lambda x: (x + 255) // 256 * 256  # noqa: E731
        tiles = s.num_tiles
        w = up(256 + 4 * tiles)
        w = up(w + 8 * (tiles + 1))
        bins = [b for specs in (k, v) for (a, e, b) in specs for _ in range(a, e)]
        nib = _count_layout(C, 16)[0] == 4 and C % 32 == 0
        row_bytes = sum(C // 2 if (nib and b == 16) else C for b in bins)
        w = up(w + T * row_bytes)
        w = up(w + 2 * L * T * ((C + 32 + 15) // 16 * 16))
        assert s.workspace_bytes == w
    finally:
        cg.cg_plan_destroy(plan)
