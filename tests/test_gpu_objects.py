"""Per-object containers on the GPU: one encode of every chunk_tokens
object of a blob, cut into one container per object, must give exactly the
oracle's container of each object's tokens encoded alone; and the
containers of all objects, put back with cg_deserialize_objects, must decode
in one cg_decode to the oracle's output."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

from kv_cache_compression_03_gb300 import cachegen as cg  # noqa: E402
from kv_cache_compression_03_gb300 import synthetic  # noqa: E402


def _bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("name,T,chunk", [("mistral7b_chunk_sweep", 768, 64),
                                          ("mistral7b_chunk_sweep", 768, 128),
                                          ("mistral7b_chunk_sweep", 768, 256),
                                          ("mistral7b_chunk_sweep", 768, 768),
                                          ("opt125m_t256", 700, 300)])
def test_objects_match_slices(orc, name, T, chunk):
    p = synthetic.WORKLOADS[name]
    H, D = p["H"], p["D"]
    bits = synthetic.generate(name, num_tokens=T)
    k, v = synthetic.workload_specs(name)
    L, _, T, C = bits.shape
    codec = cg.Codec(L, T, H, D, chunk, k, v)
    kv = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).reshape(L, 2, T, H, D).cuda()
    enc = codec.encode(kv)
    objs = codec.object_bytes(enc)
    assert len(objs) == codec.sizes.num_objects == -(-T // chunk)
    offset = 0
    for o, blob in enumerate(objs):
        t0, n = cg.cg_object_range(codec.plan, o)
        part = np.ascontiguousarray(bits[:, :, t0:t0 + n])
        ref = orc.encode(part, chunk, k, v)
        want = orc.serialize(ref, L, n, H, D, chunk, k, v)
        assert bytes(blob.numpy()) == want, o
        off, nb = cg.cg_object_streams(codec.plan, codec.workspace, o)
        assert (off, nb) == (offset, ref["stream_bytes"])
        offset += nb
    assert offset == enc.stream_bytes
    # all objects back into one blob, one decode
    enc2 = codec.from_object_bytes(objs)
    assert enc2.stream_bytes == enc.stream_bytes
    n = enc.stream_bytes
    assert torch.equal(enc2.bytestream[:n], enc.bytestream[:n])
    assert torch.equal(enc2.lengths, enc.lengths) and torch.equal(enc2.cdf, enc.cdf)
    assert torch.equal(enc2.amax, enc.amax)
    out = codec.decode(enc2)
    full = orc.encode(bits, chunk, k, v)
    assert np.array_equal(_bits(out).reshape(L, 2, T, C), orc.decode(full, L, T, C, chunk, k, v))
