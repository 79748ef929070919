"""GPU parity: the CUDA codec (through the C ABI) against the CPU oracle on
the same seeded inputs. Symbols, scales, CDF tables, stream lengths and
packed bytes must be bit-exact; decoded bf16 must be within 1 bf16 ulp of
the oracle (and is checked bit-exact too, since both evaluate the same
fp32 operations in the same order)."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

from kv_cache_compression_03_gb300 import cachegen as cg  # noqa: E402
from kv_cache_compression_03_gb300 import synthetic  # noqa: E402


def _to_dev(bits: np.ndarray, H: int, D: int):
    L, _, T, C = bits.shape
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return t.reshape(L, 2, T, H, D).cuda()


def _bits(t) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _ulp_diff(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    # ordered integer view of bf16 bit patterns
    def key(x):
        x = x.astype(np.int32)
        return np.where(x & 0x8000, 0x8000 - (x & 0x7FFF), 0x8000 + (x & 0x7FFF))
    return np.abs(key(a) - key(b))


def _run(bits, H, D, chunk, k, v):
    L, _, T, C = bits.shape
    codec = cg.Codec(L, T, H, D, chunk, k, v)
    kv = _to_dev(bits, H, D)
    enc = codec.encode(kv)
    out = codec.decode(enc)
    torch.cuda.synchronize()
    return codec, kv, enc, out


def _compare(orc, bits, H, D, chunk, k, v):
    L, _, T, C = bits.shape
    codec, kv, enc, out = _run(bits, H, D, chunk, k, v)
    ref = orc.encode(bits, chunk, k, v)
    assert np.array_equal(enc.amax.cpu().numpy(), ref["amax"])
    assert np.array_equal(enc.cdf.cpu().numpy().view(np.uint16), ref["cdf"])
    assert np.array_equal(enc.lengths.cpu().numpy(), ref["lengths"])
    assert enc.stream_bytes == ref["stream_bytes"]
    assert np.array_equal(enc.bytestream[:enc.stream_bytes].cpu().numpy(), ref["bytes"])
    want, sym = orc.decode(ref, L, T, C, chunk, k, v, want_symbols=True)
    got = _bits(out).reshape(L, 2, T, C)
    assert _ulp_diff(got, want).max() <= 1          # the stated tolerance
    assert np.array_equal(got, want)                 # and in fact bit-exact
    return codec, enc, ref, got


CASES = [
    ("opt125m_t256", None, 256),
    ("opt125m_t256", 300, 256),            # ragged second group (44 tokens)
    ("mistral7b_t1k", None, 256),
    ("mistral7b_chunk_sweep", None, 64),
    ("mistral7b_chunk_sweep", None, 128),
    ("mistral7b_chunk_sweep", None, 256),
    ("mistral7b_chunk_sweep", None, 768),
    ("llama8b_t16k", 700, 256),            # heavy tails + token spikes, ragged
    ("glm4_9b_t32k", 1100, 256),           # C = 256, ragged
]


@pytest.mark.parametrize("name,T,chunk", CASES, ids=[f"{c[0]}-{c[1]}-{c[2]}" for c in CASES])
def test_parity_workloads(orc, name, T, chunk):
    p = synthetic.WORKLOADS[name]
    bits = synthetic.generate(name, num_tokens=T)
    k, v = synthetic.workload_specs(name)
    _compare(orc, bits, p["H"], p["D"], chunk, k, v)


def test_reconstruction_bound():
    name = "mistral7b_t1k"
    p = synthetic.WORKLOADS[name]
    bits = synthetic.generate(name, num_tokens=512)
    k, v = synthetic.workload_specs(name)
    codec, kv, enc, out = _run(bits, p["H"], p["D"], 256, k, v)
    L, _, T, C = bits.shape
    x = kv.float().reshape(L, 2, T, C).permute(1, 0, 2, 3).double()
    y = out.float().reshape(L, 2, T, C).permute(1, 0, 2, 3).double()
    bins = torch.tensor([[32 if l < 10 else 16 for l in range(L)],
                         [32 if l < 2 else 16 for l in range(L)]], dtype=torch.float64).cuda()
    M = (bins / 2 - 1)[:, :, None, None]
    a = enc.amax.double()[..., None]
    bound = 0.5 * a / M * (1 + 2.0 ** -20) + y.abs() * 2.0 ** -8
    assert bool(((x - y).abs() <= bound).all())


EDGE = [
    # (L, T, H, D, chunk, kspecs, vspecs, generator)
    (2, 1, 1, 8, 256, [(0, 2, 16)], [(0, 2, 32)], "normal"),        # one token
    (3, 257, 2, 8, 256, [(0, 3, 4)], [(0, 3, 64)], "normal"),       # 4 and 64 bins
    (2, 40, 1, 16, 1, [(0, 2, 16)], [(0, 2, 16)], "normal"),        # groups of 1 token
    (4, 700, 1, 64, 300, [(0, 1, 8), (1, 4, 30)], [(0, 4, 12)], "normal"),
    (2, 300, 2, 32, 256, [(0, 2, 32)], [(0, 2, 16)], "zeros"),      # all-zero rows
    (2, 300, 2, 32, 256, [(0, 2, 32)], [(0, 2, 16)], "constant"),   # one value per row
    (2, 300, 2, 32, 256, [(0, 2, 32)], [(0, 2, 16)], "extreme"),    # huge and tiny values
    (1, 513, 8, 64, 1000, [(0, 1, 64)], [(0, 1, 4)], "normal"),     # chunk > T
    (2, 64, 8, 512, 64, [(0, 2, 16)], [(0, 2, 16)], "normal"),      # C = 4096 (16 bins)
    (2, 100, 16, 128, 64, [(0, 2, 32)], [(0, 1, 16), (1, 2, 32)], "normal"),  # C = 2048
    (2, 256, 4, 64, 256, [(0, 2, 32)], [(0, 2, 16)], "bimodal"),    # near-half CDF splits
    (2, 300, 2, 32, 256, [(0, 2, 64)], [(0, 2, 16)], "tiny"),       # amax near 2^-118
    (2, 512, 2, 64, 256, [(0, 2, 16)], [(0, 2, 32)], "sparse"),     # rows of rare symbols only
    (1, 256, 1, 64, 256, [(0, 1, 16)], [(0, 1, 16)], "sparse1"),    # one busy row per group
    # C >= 1024 and a multiple of 32: 16-bin symbols kept as 4-bit codes
    (2, 300, 8, 128, 256, [(0, 2, 16)], [(0, 2, 32)], "sparse"),    # 4-bit codes, exact re-code
    (2, 256, 8, 128, 256, [(0, 2, 16)], [(0, 2, 16)], "bimodal"),   # 4-bit codes, carry runs
    (1, 300, 8, 160, 256, [(0, 1, 16)], [(0, 1, 16)], "extreme"),   # C = 1280, ragged group
    (1, 100, 3, 344, 256, [(0, 1, 16)], [(0, 1, 16)], "normal"),    # C = 1032: byte codes
    # CDF tables above the shared-memory budget, coded and decoded in channel
    # parts: 64 bins (4 parts), 48 bins (3 parts, the last one shorter)
    (1, 300, 8, 128, 256, [(0, 1, 64)], [(0, 1, 48)], "normal"),
    (1, 300, 8, 128, 256, [(0, 1, 64)], [(0, 1, 32)], "sparse"),    # parts + exact re-codes
    (1, 260, 8, 128, 256, [(0, 1, 64)], [(0, 1, 32)], "bimodal"),   # parts + carry runs
    (1, 64, 32, 128, 64, [(0, 1, 32)], [(0, 1, 64)], "normal"),     # C = 4096: 8 and 15 parts
    # rows under 1024 channels counted by row groups into private histograms
    (2, 300, 1, 128, 256, [(0, 2, 16)], [(0, 2, 32)], "normal"),    # C = 128: 8 / 4 groups
    (2, 300, 1, 64, 256, [(0, 2, 16)], [(0, 2, 8)], "sparse"),      # C = 64: 8 groups of 32
    (1, 300, 4, 128, 256, [(0, 1, 16)], [(0, 1, 32)], "extreme"),   # C = 512: 2 groups
]


def _edge_bits(L, T, C, kind, seed):
    rng = np.random.default_rng(seed)
    if kind == "zeros":
        b = np.zeros((L, 2, T, C), dtype=np.uint16)
        b[..., ::3] = 0x8000  # -0.0 too
        return b
    if kind == "bimodal":
        # every value is +-1: symbols 0 and 2*MAX with near-equal counts, so the
        # coder's interval keeps straddling the middle (long pending runs, carries)
        x = np.where(rng.random((L, 2, T, C)) < 0.5, -1.0, 1.0)
    elif kind == "constant":
        x = np.broadcast_to(rng.standard_normal((L, 2, T, 1)), (L, 2, T, C))
    elif kind in ("sparse", "sparse1"):
        # most token rows are zero (every symbol is MAX); a few rows hold
        # values, so each of their symbols occurs once or twice in its
        # channel's group: ~8-9 bits per symbol, which fills the coders' bit
        # buffers between checks
        x = np.zeros((L, 2, T, C))
        busy = [37] if kind == "sparse1" else [3, 100, 101, 255, 300, 511]
        for t in busy:
            if t < T:
                x[:, :, t, :] = rng.standard_normal((L, 2, C))
    elif kind == "tiny":
        # rows just above the smallest amax with a finite MAX / a
        x = rng.standard_normal((L, 2, T, C)) * 2.0 ** -118
    elif kind == "extreme":
        x = rng.standard_normal((L, 2, T, C)) * np.exp(rng.uniform(-80, 80, (L, 2, T, 1)))
        x[..., 0] = 3.0e38
        x[:, :, 1::2, 1] = 1e-38
    else:
        x = rng.standard_normal((L, 2, T, C))
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


@pytest.mark.parametrize("case", EDGE, ids=[f"edge{i}" for i in range(len(EDGE))])
def test_parity_edges(orc, case):
    L, T, H, D, chunk, k, v, kind = case
    bits = _edge_bits(L, T, H * D, kind, seed=L * 1000 + T)
    _compare(orc, bits, H, D, chunk, k, v)


def test_serialize_matches_oracle_container(orc):
    name = "opt125m_t256"
    p = synthetic.WORKLOADS[name]
    bits = synthetic.generate(name, num_tokens=600)
    k, v = synthetic.workload_specs(name)
    L, _, T, C = bits.shape
    codec, kv, enc, out = _run(bits, p["H"], p["D"], 256, k, v)
    blob = codec.to_bytes(enc)
    ref = orc.encode(bits, 256, k, v)
    want = orc.serialize(ref, L, T, p["H"], p["D"], 256, k, v)
    assert bytes(blob.numpy()) == want
    # and back: open, copy to the device, decode
    codec2, enc2 = cg.Codec.from_bytes(blob)
    out2 = codec2.decode(enc2)
    assert np.array_equal(_bits(out2), _bits(out))


def test_container_copies_through_every_kind_of_host_buffer(orc):
    """cg_serialize / cg_deserialize with pinned and pageable host buffers, at
    offsets of 0, 4 and 1 bytes from an aligned start: every form gives the
    oracle's container and decodes it back."""
    name = "mistral7b_t1k"
    p = synthetic.WORKLOADS[name]
    bits = synthetic.generate(name, num_tokens=300)
    k, v = synthetic.workload_specs(name)
    L, _, T, C = bits.shape
    codec, kv, enc, out = _run(bits, p["H"], p["D"], 256, k, v)
    ref = orc.encode(bits, 256, k, v)
    want = orc.serialize(ref, L, T, p["H"], p["D"], 256, k, v)
    n = len(want)
    pinned = torch.empty(n + 64, dtype=torch.uint8, pin_memory=True)
    pageable = torch.empty(n + 64, dtype=torch.uint8)
    for buf in (pinned, pageable):
        for off in (0, 4, 1):
            host = buf[off:off + n]
            host.fill_(0xA5)
            w = cg.cg_serialize(codec.plan, enc.bytestream, enc.lengths, enc.cdf, enc.amax,
                                enc.stream_bytes, host)
            assert w == n
            assert bytes(host.numpy()) == want, (buf.is_pinned(), off)
            enc2 = codec.alloc_encoded()
            cg.cg_deserialize(codec.plan, host, enc2.bytestream, enc2.lengths, enc2.cdf,
                              enc2.amax)
            enc2.stream_bytes = enc.stream_bytes
            out2 = codec.decode(enc2)
            torch.cuda.synchronize()
            assert np.array_equal(_bits(out2), _bits(out)), (buf.is_pinned(), off)


def test_repeatable_and_side_stream(orc):
    name = "mistral7b_t1k"
    p = synthetic.WORKLOADS[name]
    bits = synthetic.generate(name, num_tokens=300)
    k, v = synthetic.workload_specs(name)
    L, _, T, C = bits.shape
    codec = cg.Codec(L, T, p["H"], p["D"], 256, k, v)
    kv = _to_dev(bits, p["H"], p["D"])
    a = codec.encode(kv)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        b = codec.encode(kv, stream=s)
        out = codec.decode(b, stream=s)
    s.synchronize()
    n = a.stream_bytes
    assert n == b.stream_bytes
    assert torch.equal(a.bytestream[:n], b.bytestream[:n])
    assert torch.equal(a.lengths, b.lengths) and torch.equal(a.cdf, b.cdf)
    ref = orc.encode(bits, 256, k, v)
    assert np.array_equal(_bits(out).reshape(L, 2, T, C), orc.decode(ref, L, T, C, 256, k, v))


@pytest.mark.parametrize("name,T", [("mistral7b_t1k", 300), ("llama8b_t16k", 300)])
def test_decode_into_an_output_aligned_to_16_bytes_only(orc, name, T):
    """The decoder writes 32-byte sectors when the output allows it; an
    output that starts 16 bytes past a 32-byte boundary takes the kernels
    with 16-byte stores (llama: 16-bin tiles and 32-bin tiles in channel
    parts). Both must give the oracle's bytes."""
    p = synthetic.WORKLOADS[name]
    bits = synthetic.generate(name, num_tokens=T)
    k, v = synthetic.workload_specs(name)
    L, _, T, C = bits.shape
    codec = cg.Codec(L, T, p["H"], p["D"], 256, k, v)
    enc = codec.encode(_to_dev(bits, p["H"], p["D"]))
    n = L * 2 * T * C
    buf = torch.empty(n + 32, dtype=torch.bfloat16, device="cuda")
    off = ((32 - buf.data_ptr() % 32) % 32 + 16) // 2
    out = buf[off:off + n].view(L, 2, T, p["H"], p["D"])
    assert out.data_ptr() % 32 == 16
    codec.decode(enc, kv_out=out)
    ref = orc.encode(bits, 256, k, v)
    want = orc.decode(ref, L, T, C, 256, k, v)
    assert np.array_equal(_bits(out).reshape(L, 2, T, C), want)
    aligned = codec.decode(enc)
    assert aligned.data_ptr() % 32 == 0
    assert np.array_equal(_bits(aligned).reshape(L, 2, T, C), want)


def test_nonfinite_input_is_reported():
    name = "opt125m_t256"
    p = synthetic.WORKLOADS[name]
    bits = synthetic.generate(name, num_tokens=64).copy()
    bits[3, 1, 17, 5] = 0x7F80    # +inf
    bits[0, 0, 2, 100] = 0x7FC1   # NaN
    k, v = synthetic.workload_specs(name)
    L, _, T, C = bits.shape
    codec = cg.Codec(L, T, p["H"], p["D"], 256, k, v)
    kv = _to_dev(bits, p["H"], p["D"])
    enc = codec.alloc_encoded()
    cg.cg_encode(codec.plan, kv, codec.workspace, enc.bytestream, enc.lengths, enc.cdf, enc.amax)
    st, total = cg.cg_last_device_error(codec.plan, codec.workspace)
    assert st == cg.CG_ERR_NONFINITE
    assert 0 < total <= codec.sizes.max_stream_bytes


def test_nonfinite_rows_with_4bit_codes_are_reported():
    # 1024-channel rows (16-bin symbols kept as 4-bit codes): a row of NaN,
    # scattered infinities; the status is reported and every stream stays
    # inside its bounds (the output itself is undefined)
    name = "llama8b_t16k"
    p = synthetic.WORKLOADS[name]
    bits = synthetic.generate(name, num_tokens=300).copy()
    bits[20, 0, 7, :] = 0x7FC0          # a whole K row of NaN (16 bins)
    bits[20, 1, 260, ::97] = 0xFF80     # -inf in a V row (16 bins)
    bits[1, 0, 3, 5] = 0x7F80           # +inf in a 32-bin row
    k, v = synthetic.workload_specs(name)
    L, _, T, C = bits.shape
    codec = cg.Codec(L, T, p["H"], p["D"], 256, k, v)
    enc = codec.alloc_encoded()
    cg.cg_encode(codec.plan, _to_dev(bits, p["H"], p["D"]), codec.workspace, enc.bytestream,
                 enc.lengths, enc.cdf, enc.amax)
    st, total = cg.cg_last_device_error(codec.plan, codec.workspace)
    assert st == cg.CG_ERR_NONFINITE
    lengths = enc.lengths.cpu().numpy()
    assert lengths.min() >= 1 and lengths.max() <= 3 * C


def test_tiny_row_is_reported():
    # a row whose amax (2^-126) makes MAX / a overflow fp32 has no scale factor
    name = "opt125m_t256"
    p = synthetic.WORKLOADS[name]
    bits = synthetic.generate(name, num_tokens=64).copy()
    bits[2, 0, 9, :] = 0
    bits[2, 0, 9, 7] = 0x0080
    k, v = synthetic.workload_specs(name)
    L, _, T, C = bits.shape
    codec = cg.Codec(L, T, p["H"], p["D"], 256, k, v)
    enc = codec.alloc_encoded()
    cg.cg_encode(codec.plan, _to_dev(bits, p["H"], p["D"]), codec.workspace, enc.bytestream,
                 enc.lengths, enc.cdf, enc.amax)
    st, _ = cg.cg_last_device_error(codec.plan, codec.workspace)
    assert st == cg.CG_ERR_NONFINITE


def test_capacity_too_small_is_reported_without_overrun(orc):
    name = "opt125m_t256"
    p = synthetic.WORKLOADS[name]
    bits = synthetic.generate(name, num_tokens=256)
    k, v = synthetic.workload_specs(name)
    L, _, T, C = bits.shape
    need = orc.encode(bits, 256, k, v)["stream_bytes"]
    codec = cg.Codec(L, T, p["H"], p["D"], 256, k, v)
    kv = _to_dev(bits, p["H"], p["D"])
    cap = (need // 2) // 16 * 16
    big = torch.full((cap + 4096,), 0xA5, dtype=torch.uint8, device="cuda")
    enc = codec.alloc_encoded()
    cg.cg_encode(codec.plan, kv, codec.workspace, big[:cap], enc.lengths, enc.cdf, enc.amax)
    st, total = cg.cg_last_device_error(codec.plan, codec.workspace)
    assert st == cg.CG_ERR_CAPACITY
    assert total == need
    assert bool((big[cap:] == 0xA5).all())


def test_corrupt_containers_are_reported(orc):
    name = "opt125m_t256"
    p = synthetic.WORKLOADS[name]
    bits = synthetic.generate(name, num_tokens=300)
    k, v = synthetic.workload_specs(name)
    L, _, T, C = bits.shape
    codec, kv, enc, out = _run(bits, p["H"], p["D"], 256, k, v)

    def decode_status(e, sb=None):
        o = torch.empty_like(out)
        cg.cg_decode(codec.plan, e.bytestream, e.lengths, e.cdf, e.amax,
                     e.stream_bytes if sb is None else sb, codec.workspace, o)
        return cg.cg_last_device_error(codec.plan, codec.workspace)[0], o

    base = cg.Encoded(enc.bytestream.clone(), enc.lengths.clone(), enc.cdf.clone(),
                      enc.amax.clone(), enc.stream_bytes)
    assert decode_status(base)[0] == cg.CG_OK
    # flipped stream bits: decoding ends normally, the output changes
    e1 = cg.Encoded(base.bytestream.clone(), base.lengths, base.cdf, base.amax, base.stream_bytes)
    e1.bytestream[100:140] ^= 0x5A
    st, o1 = decode_status(e1)
    assert st == cg.CG_OK and not torch.equal(o1, out)
    # a CDF row that does not rise strictly
    e2 = cg.Encoded(base.bytestream, base.lengths, base.cdf.clone(), base.amax, base.stream_bytes)
    e2.cdf[5] = e2.cdf[4]
    assert decode_status(e2)[0] == cg.CG_ERR_CORRUPT
    # lengths that do not add up to the stream size
    e3 = cg.Encoded(base.bytestream, base.lengths.clone(), base.cdf, base.amax, base.stream_bytes)
    e3.lengths[7] += 3
    assert decode_status(e3)[0] == cg.CG_ERR_CORRUPT
    e4 = cg.Encoded(base.bytestream, base.lengths.clone(), base.cdf, base.amax, base.stream_bytes)
    e4.lengths[9] = -5
    assert decode_status(e4)[0] == cg.CG_ERR_CORRUPT
    assert decode_status(base, sb=base.stream_bytes - 16)[0] == cg.CG_ERR_CORRUPT


@pytest.mark.parametrize("H,D,N", [(1, 32, 16), (8, 128, 32), (8, 128, 64)])
def test_decoder_batches_that_run_short(orc, H, D, N):
    """The decoder refills its bit buffer once per few symbols; a run of
    symbols of frequency 1/65536 (which this encoder never produces, but a
    valid container may hold) takes ~16 bits each, so such a batch runs short
    and the stream (or, where the CDF table is staged in channel parts: 32
    and 64 bins at 1024 channels, that part) is decoded again exactly. Built
    by hand: CDF rows with two frequency-1 symbols, streams coded by the
    oracle's coder."""
    L, T = 1, 64
    C = H * D
    rng = np.random.default_rng(77)
    row = np.zeros(N + 1, dtype=np.int64)
    row[1], row[2] = 1, 2
    row[2:] = 2 + np.round(np.arange(N - 1) * (65534 / (N - 2))).astype(np.int64)
    row[N] = 65536
    assert np.all(np.diff(row) >= 1) and row[2] == 2
    rows = np.broadcast_to(row, (C, N + 1)).astype(np.uint32)
    streams, lengths = [], []
    syms = np.zeros((2, L, T, C), dtype=np.uint8)
    for kv in range(2):
        for t in range(T):
            s = rng.integers(2, N - 1, C)              # common symbols 2..14
            if t % 3 == 0:
                s[: C // 2] = rng.integers(0, 2, C // 2)  # a run of the rare ones
            elif t % 3 == 1:
                s[5:9] = 0                              # one rare batch
            syms[kv, 0, t] = s
            b = orc.wnc_encode(s, rows)
            streams.append(b)
            lengths.append(len(b))
    wire = np.tile(row.astype(np.uint32) & 0xFFFF, (2 * C, 1)).astype(np.uint16).ravel()
    enc = {"amax": rng.uniform(0.5, 2.0, (2, L, T)).astype(np.float32),
           "lengths": np.array(lengths, dtype=np.int32), "cdf": wire,
           "bytes": np.frombuffer(b"".join(streams), dtype=np.uint8),
           "stream_bytes": sum(lengths)}
    k = v = [(0, L, N)]
    want, sym = orc.decode(enc, L, T, C, 256, k, v, want_symbols=True)
    assert np.array_equal(sym, syms)
    blob = orc.serialize(enc, L, T, H, D, 256, k, v)
    codec, e = cg.Codec.from_bytes(torch.from_numpy(np.frombuffer(blob, np.uint8).copy()))
    out = codec.decode(e)
    assert np.array_equal(_bits(out).reshape(L, 2, T, C), want)


def test_encode_decode_in_a_cuda_graph(orc):
    """cg_encode and cg_decode (side-stream fork and join included) are
    stream-ordered only, so they can be captured into a CUDA graph; replays
    give the eager results."""
    name = "mistral7b_t1k"
    p = synthetic.WORKLOADS[name]
    bits = synthetic.generate(name, num_tokens=300)
    k, v = synthetic.workload_specs(name)
    L, _, T, C = bits.shape
    codec, kv, enc, out = _run(bits, p["H"], p["D"], 256, k, v)  # eager, and first-use setup
    n = enc.stream_bytes
    enc2 = codec.alloc_encoded()
    out2 = torch.empty_like(out)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        cg.cg_encode(codec.plan, kv, codec.workspace, enc2.bytestream, enc2.lengths, enc2.cdf,
                     enc2.amax)
        cg.cg_decode(codec.plan, enc2.bytestream, enc2.lengths, enc2.cdf, enc2.amax, n,
                     codec.workspace, out2)
    for _ in range(2):
        out2.zero_()
        enc2.bytestream.zero_()
        g.replay()
        torch.cuda.synchronize()
        st, total = cg.cg_last_device_error(codec.plan, codec.workspace)
        assert st == cg.CG_OK and total == n
        assert torch.equal(enc2.bytestream[:n], enc.bytestream[:n])
        assert torch.equal(enc2.lengths, enc.lengths) and torch.equal(enc2.cdf, enc.cdf)
        assert torch.equal(out2, out)
    ref = orc.encode(bits, 256, k, v)
    assert np.array_equal(_bits(out2).reshape(L, 2, T, C), orc.decode(ref, L, T, C, 256, k, v))
