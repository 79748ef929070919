"""cg_encode_noalloc: the encoder entry point for callers that cannot
allocate device memory when they encode (a serving engine whose KV cache
pool already holds nearly all of the GPU, or a latency-critical path where
cudaMalloc/cudaFree could synchronise the device). It uses the library's
fixed scratch array instead of a caller workspace. Here it is called
through the C ABI twice in a row and must give exactly what cg_encode
gives; a plan too large for the array must be refused.

This file sorts last so that a run stopping at its first failure has
already run every other test."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

from kv_cache_compression_03_gb300 import cachegen as cg  # noqa: E402
from kv_cache_compression_03_gb300 import synthetic  # noqa: E402


def _kv(name, T):
    p = synthetic.WORKLOADS[name]
    bits = synthetic.generate(name, num_tokens=T)
    L = p["L"]
    t = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16)
    return t.reshape(L, 2, T, p["H"], p["D"]).cuda(), p


def test_noalloc_matches_cg_encode_twice():
    name = "opt125m_t256"
    kv, p = _kv(name, 300)
    k, v = synthetic.workload_specs(name)
    codec = cg.Codec(p["L"], 300, p["H"], p["D"], 256, k, v)
    assert codec.sizes.workspace_bytes <= 64 * 1024 * 1024
    ref = codec.encode(kv)   # the existing entry point, with a workspace
    n = ref.stream_bytes

    status = torch.empty(16, dtype=torch.uint8, device="cuda")
    for call in range(2):
        out = codec.alloc_encoded()
        for t in (out.bytestream, out.lengths, out.cdf, out.amax):
            t.view(torch.uint8).fill_(0x5A)   # stale contents must not leak through
        cg.cg_encode_noalloc(codec.plan, kv, out.bytestream, out.lengths, out.cdf, out.amax,
                             status)
        st, total = cg.cg_last_device_error(codec.plan, status)
        assert st == cg.CG_OK, (call, st)
        assert total == n
        assert torch.equal(out.bytestream[:n], ref.bytestream[:n])
        assert torch.equal(out.lengths, ref.lengths)
        assert torch.equal(out.cdf, ref.cdf)
        assert torch.equal(out.amax, ref.amax)
        out.stream_bytes = total
        dec = codec.decode(out)
        assert torch.equal(dec.view(torch.int16), codec.decode(ref).view(torch.int16))


def test_noalloc_rejects_plans_beyond_the_scratch():
    name = "mistral7b_t1k"     # workspace ~135 MB > 64 MiB
    kv, p = _kv(name, 1024)
    k, v = synthetic.workload_specs(name)
    codec = cg.Codec(p["L"], 1024, p["H"], p["D"], 256, k, v)
    assert codec.sizes.workspace_bytes > 64 * 1024 * 1024
    out = codec.alloc_encoded()
    status = torch.zeros(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(cg.CacheGenError) as e:
        cg.cg_encode_noalloc(codec.plan, kv, out.bytestream, out.lengths, out.cdf, out.amax,
                             status)
    assert e.value.status == cg.CG_ERR_UNSUPPORTED
