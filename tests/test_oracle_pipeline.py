"""Whole-pipeline pins of the CPU oracle: round trip, reconstruction bound,
entropy bounds on the coded size, CDF-table invariants, container layout,
and agreement between the tile-sampled and whole-blob encoders."""
import struct

import numpy as np
import pytest

from kv_cache_compression_03_gb300 import synthetic


def _bf16_to_f64(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _layout(orc, L, T, chunk, kspecs, vspecs):
    kb, vb = orc.layer_bins(L, kspecs), orc.layer_bins(L, vspecs)
    gs, gc = orc.groups(T, chunk)
    return np.stack([kb, vb]), gs, gc


def _case(name, T=None, chunk=None):
    kv = synthetic.generate(name, num_tokens=T)
    k, v = synthetic.workload_specs(name)
    ch = chunk or synthetic.WORKLOADS[name]["chunk_tokens"][0]
    return kv, k, v, ch


CASES = [
    ("opt125m_t256", None, None),
    ("mistral7b_t1k", 512, None),
    ("mistral7b_chunk_sweep", 768, 64),
    ("mistral7b_chunk_sweep", 768, 768),
    ("llama8b_t16k", 300, None),
    ("glm4_9b_t32k", 600, None),
]


@pytest.fixture(scope="module", params=CASES, ids=lambda c: f"{c[0]}-{c[1]}-{c[2]}")
def encoded(request, orc):
    name, T, chunk = request.param
    kv, k, v, ch = _case(name, T, chunk)
    enc = orc.encode(kv, ch, k, v, want_symbols=True)
    return kv, k, v, ch, enc


def test_roundtrip_and_reconstruction(orc, encoded):
    kv, k, v, ch, enc = encoded
    L, _, T, C = kv.shape
    out, sym = orc.decode(enc, L, T, C, ch, k, v, want_symbols=True)
    assert np.array_equal(sym, enc["symbols"])
    bins, _, _ = _layout(orc, L, T, ch, k, v)
    M = (bins // 2 - 1).astype(np.float64)  # [2, L]
    x = _bf16_to_f64(kv.transpose(1, 0, 2, 3))      # [2, L, T, C]
    y = _bf16_to_f64(out.transpose(1, 0, 2, 3))
    a = enc["amax"].astype(np.float64)[..., None]   # [2, L, T, 1]
    step = a / M[:, :, None, None]
    err = np.abs(x - y)
    assert np.all(err <= 0.5 * step * (1 + 2.0 ** -20) + np.abs(y) * 2.0 ** -8 + 1e-30)
    # amax is the exact max |x| per (kv, layer, token)
    assert np.array_equal(enc["amax"].astype(np.float64), np.abs(x).max(axis=-1))


def test_cdf_tables_match_histograms(orc, encoded):
    kv, k, v, ch, enc = encoded
    L, _, T, C = kv.shape
    bins, gs, gc = _layout(orc, L, T, ch, k, v)
    sym = enc["symbols"]
    cdf = enc["cdf"].astype(np.int64)
    off = 0
    for g in range(len(gs)):
        for kvs in range(2):
            for l in range(L):
                N = int(bins[kvs, l])
                blk = cdf[off:off + C * (N + 1)].reshape(C, N + 1)
                off += C * (N + 1)
                assert np.all(blk[:, 0] == 0) and np.all(blk[:, N] == 0)
                full = blk.copy()
                full[:, N] = 65536
                freq = np.diff(full, axis=1)
                assert np.all(freq >= 1) and np.all(freq.sum(axis=1) == 65536)
                s = sym[kvs, l, gs[g]:gs[g] + gc[g]]            # [n, C]
                counts = np.zeros((C, N), dtype=np.int64)
                np.add.at(counts, (np.broadcast_to(np.arange(C), s.shape), s), 1)
                assert np.array_equal(freq == 1, counts == 0)
                share = counts * (65536 - N) / gc[g]
                assert np.all(np.abs((freq - 1) - share) < 1.0)
    assert off == cdf.size


def test_coded_size_entropy_bounds(orc, encoded):
    """Coded bits lie between the cross-entropy under the integer CDFs and
    that plus 2 bits (+ padding) per stream; and within 1 % (+ the same
    per-stream terms) of the empirical per-channel entropy of each group."""
    kv, k, v, ch, enc = encoded
    L, _, T, C = kv.shape
    bins, gs, gc = _layout(orc, L, T, ch, k, v)
    sym = enc["symbols"]
    cdf = enc["cdf"].astype(np.int64)
    lengths = enc["lengths"].astype(np.int64)
    off = 0
    cross = 0.0
    h_emp = 0.0
    si = 0
    for g in range(len(gs)):
        n = int(gc[g])
        for kvs in range(2):
            for l in range(L):
                N = int(bins[kvs, l])
                full = cdf[off:off + C * (N + 1)].reshape(C, N + 1).copy()
                off += C * (N + 1)
                full[:, N] = 65536
                freq = np.diff(full, axis=1)
                s = sym[kvs, l, gs[g]:gs[g] + n].astype(np.int64)
                f_used = freq[np.arange(C)[None, :], s]
                bits_tok = np.sum(16 - np.log2(f_used), axis=1)        # per stream
                stream_bits = 8 * lengths[si:si + n]
                assert np.all(stream_bits >= bits_tok - C * 2.0 ** -13 - 1e-6)
                assert np.all(stream_bits <= bits_tok + 2 + 7 + C * 2.0 ** -13 + 1e-6)
                cross += bits_tok.sum()
                counts = np.zeros((C, N), dtype=np.int64)
                np.add.at(counts, (np.broadcast_to(np.arange(C), s.shape), s), 1)
                p = counts / n
                with np.errstate(divide="ignore", invalid="ignore"):
                    h_emp += -np.nansum(counts * np.log2(np.where(p > 0, p, 1)))
                si += n
    total_bits = 8 * int(lengths.sum())
    assert total_bits == 8 * enc["stream_bytes"]
    S = 2 * L * T
    assert total_bits <= 1.01 * h_emp + 9 * S
    assert total_bits >= h_emp - 1e-6 * S


def test_tiles_match_whole(orc, encoded):
    kv, k, v, ch, enc = encoded
    L, _, T, C = kv.shape
    bins, gs, gc = _layout(orc, L, T, ch, k, v)
    ntiles = len(gs) * 2 * L
    pick = sorted({0, ntiles - 1, ntiles // 2, 1 % ntiles, (7 * ntiles) // 9})
    got = orc.encode_tiles(kv, ch, k, v, pick)
    # offsets of tiles in the whole blob
    cdf_off, stream_first, byte_off = [], [], []
    co, sf, bo = 0, 0, 0
    lengths = enc["lengths"].astype(np.int64)
    for g in range(len(gs)):
        for kvs in range(2):
            for l in range(L):
                cdf_off.append(co)
                stream_first.append(sf)
                byte_off.append(bo)
                co += C * (int(bins[kvs, l]) + 1)
                n = int(gc[g])
                bo += int(lengths[sf:sf + n].sum())
                sf += n
    for t in got:
        ti = t["tile"]
        g, kvs, l = ti // (2 * L), (ti // L) % 2, ti % L
        n = int(gc[g])
        N = int(bins[kvs, l])
        assert np.array_equal(t["cdf"], enc["cdf"][cdf_off[ti]:cdf_off[ti] + C * (N + 1)])
        assert np.array_equal(t["lengths"], enc["lengths"][stream_first[ti]:stream_first[ti] + n])
        assert np.array_equal(t["amax"], enc["amax"][kvs, l, gs[g]:gs[g] + n])
        nb = int(t["lengths"].sum())
        assert np.array_equal(t["bytes"], enc["bytes"][byte_off[ti]:byte_off[ti] + nb])


def test_container_layout(orc):
    kv, k, v, ch = _case("opt125m_t256")
    L, _, T, C = kv.shape
    H, D = 12, 64
    enc = orc.encode(kv, ch, k, v)
    blob = orc.serialize(enc, L, T, H, D, ch, k, v)
    assert blob[:4] == b"CGKV"
    ver, L2, T2, H2, D2, ch2, nk, nv, ng, sb = struct.unpack_from("<IiiiiiiiiQ", blob, 4)
    assert (ver, L2, T2, H2, D2, ch2, nk, nv, ng) == (1, L, T, H, D, ch, len(k), len(v), 1)
    assert sb == enc["stream_bytes"]
    p = 48
    specs = struct.unpack_from(f"<{3 * (nk + nv)}i", blob, p)
    assert list(specs) == [x for s in list(k) + list(v) for x in s]
    p += 12 * (nk + nv)
    S = 2 * L * T
    assert np.array_equal(np.frombuffer(blob, np.float32, S, p), enc["amax"].ravel())
    p += 4 * S
    assert np.array_equal(np.frombuffer(blob, np.int32, S, p), enc["lengths"])
    p += 4 * S
    ne = enc["cdf"].size
    assert np.array_equal(np.frombuffer(blob, np.uint16, ne, p), enc["cdf"])
    p += 2 * ne
    assert blob[p:] == enc["bytes"].tobytes()
    # raw / container
    raw = kv.nbytes
    assert len(blob) == orc.container_size(L, T, len(k) + len(v), ne, sb)
    assert 2.0 < raw / len(blob) < 20.0
