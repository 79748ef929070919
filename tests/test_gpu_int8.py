"""GPU parity of the int8 baseline codec (cg_int8_encode / cg_int8_decode,
through the C ABI) against the oracle: bytes and scales bit-exact, decoded
bf16 bit-exact (the stated tolerance is 1 bf16 ulp; both sides evaluate the
same fp32 operations), on the workloads' shapes, ragged row lengths, every
byte value, and the degenerate rows."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

from kv_cache_compression_03_gb300 import cachegen as cg  # noqa: E402
from kv_cache_compression_03_gb300 import synthetic  # noqa: E402


def _dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def _bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _check_rows(orc, bits):
    """bits: uint16 [rows, C]."""
    rows, C = bits.shape
    x = _dev(bits)
    q, sc, _ = cg.int8_encode(x)
    y = cg.int8_decode(q, sc)
    torch.cuda.synchronize()
    rq, rs = orc.int8_encode(bits)
    assert np.array_equal(sc.cpu().numpy(), rs)
    assert np.array_equal(q.cpu().numpy(), rq)
    want = orc.int8_decode(rq, rs)
    got = _bits(y)
    assert np.array_equal(got, want)
    return q, sc, got


@pytest.mark.parametrize("name,T", [("opt125m_t256", 256), ("mistral7b_t1k", 300),
                                    ("llama8b_t16k", 129), ("glm4_9b_t32k", 77)])
def test_int8_parity_workloads(orc, name, T):
    bits = synthetic.generate(name, num_tokens=T)
    L, _, T, C = bits.shape
    _check_rows(orc, bits.reshape(-1, C))


@pytest.mark.parametrize("C", [8, 16, 248, 264, 768, 1032, 2056, 4096])
def test_int8_ragged_row_lengths(orc, C):
    rng = np.random.default_rng(C)
    x = (rng.standard_normal((37, C)) * rng.lognormal(0, 2, (37, 1))).astype(np.float32)
    u = x.view(np.uint32)
    bits = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    bits[3] = 0          # all-zero row
    bits[4, ::2] = 0x8000  # -0.0 and +0.0
    bits[4, 1::2] = 0
    _check_rows(orc, bits)


def test_int8_every_byte_decodes(orc):
    q = np.arange(256, dtype=np.uint8).view(np.int8).reshape(1, 256).repeat(5, axis=0)
    scales = np.array([1.0, 3.0e38, 1.0e-30, 0.0, 7.25], dtype=np.float32)
    y = torch.empty((5, 256), dtype=torch.bfloat16, device="cuda")
    cg.cg_int8_decode(torch.from_numpy(q).cuda(), torch.from_numpy(scales).cuda(), 5, 256, y)
    torch.cuda.synchronize()
    assert np.array_equal(_bits(y), orc.int8_decode(q, scales))


def test_int8_tiny_rows(orc):
    # rows whose amax sits just above the overflow limit of 127 / a are coded
    # like any other; below it they are reported
    rng = np.random.default_rng(5)
    x = (rng.standard_normal((16, 64)) * 2.0 ** -118).astype(np.float32)
    u = x.view(np.uint32)
    bits = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    _check_rows(orc, bits)
    bits[7] = 0x0001  # a = 2^-133, 127 / a overflows
    q, sc, st = cg.int8_encode(_dev(bits), sync=False)
    code, _ = cg.cg_last_device_error(None, st)
    assert code == cg.CG_ERR_NONFINITE


def test_int8_nonfinite_reported():
    bits = synthetic.generate("opt125m_t256", num_tokens=8).reshape(-1, 768).copy()
    for bad in (0x7F80, 0xFF80, 0x7FC0):
        b = bits.copy()
        b[5, 9] = bad
        _, _, st = cg.int8_encode(_dev(b), sync=False)
        code, _ = cg.cg_last_device_error(None, st)
        assert code == cg.CG_ERR_NONFINITE
    _, _, st = cg.int8_encode(_dev(bits), sync=False)
    assert cg.cg_last_device_error(None, st)[0] == cg.CG_OK


def test_int8_empty_and_stream(orc):
    st = torch.full((16,), 0xFF, dtype=torch.uint8, device="cuda")
    cg.cg_int8_encode(None, 0, 1024, None, None, st)
    assert cg.cg_last_device_error(None, st) == (cg.CG_OK, 0)
    cg.cg_int8_decode(None, None, 0, 1024, None)
    bits = synthetic.generate("mistral7b_t1k", num_tokens=64).reshape(-1, 1024)
    s = torch.cuda.Stream()
    x = _dev(bits)
    with torch.cuda.stream(s):
        q, sc, _ = cg.int8_encode(x, stream=s, sync=False)
        y = cg.int8_decode(q, sc, stream=s)
    s.synchronize()
    rq, rs = orc.int8_encode(bits)
    assert np.array_equal(q.cpu().numpy(), rq) and np.array_equal(_bits(y), orc.int8_decode(rq, rs))


def test_int8_full_size_sampled(orc):
    """The 16K-token Llama-8B shape in one launch: sampled rows against the
    oracle, and properties of every row."""
    bits = synthetic.generate("llama8b_t16k")
    L, _, T, C = bits.shape
    x = _dev(bits).reshape(-1, C)
    q, sc, _ = cg.int8_encode(x)
    y = cg.int8_decode(q, sc)
    torch.cuda.synchronize()
    rows = L * 2 * T
    rng = np.random.default_rng(11)
    pick = np.unique(np.concatenate([rng.integers(0, rows, 300), [0, rows - 1]]))
    flat = bits.reshape(-1, C)
    qn = q[torch.from_numpy(pick).cuda()].cpu().numpy()
    yn = _bits(y[torch.from_numpy(pick).cuda()])
    scn = sc.cpu().numpy()
    for i, r in enumerate(pick):
        a, qr = orc.int8_quantize_row(flat[r])
        assert a == scn[r] and np.array_equal(qn[i], qr)
        assert np.array_equal(yn[i], orc.int8_dequant_row(qr, a))
    # every row: amax is the row's max |x|, and some value reaches +-127
    xa = x.float().abs().amax(dim=1)
    assert torch.equal(xa, sc)
    qa = q.abs().amax(dim=1)
    assert bool(((qa == 127) | (sc == 0)).all())
