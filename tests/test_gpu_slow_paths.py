"""The rarely taken exact paths, forced on, against the oracle.

The fast paths fall back to exact ones only rarely on real data: the
decoder's search target misses a bound about once in 10^5 symbols, the
encoder redoes a stream exactly only after a carry runs through its held
word or a batch overfills its bit buffer, and the decoder redoes a stream
only when a batch of symbols runs its bit buffer short. These tests build
the library twice more with test-only macros that take those paths for
(nearly) every symbol, stream and part, and check that every output is
still the oracle's:

- CG_TEST_TARGET_MISS: every decoder search target is 0, so each symbol
  above the lowest is found by the exact re-search;
- CG_TEST_EXACT_PATHS: the encoder codes every stream again exactly (with
  channel parts: every part after the first, switching from the fast state
  mid-stream) and the decoder decodes every stream (or part) again
  refilling its bit buffer after every symbol.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

from kv_cache_compression_03_gb300 import build, cachegen as cg  # noqa: E402
from kv_cache_compression_03_gb300 import synthetic  # noqa: E402

from test_gpu_parity import _bits, _to_dev  # noqa: E402

# (workload, tokens, chunk, bins override): 16-bin 4-bit symbols and 32-bin
# channel parts at 1024 channels; 256-channel rows counted by row groups; a
# generic bin count at 1032 channels (16-byte decoder stores); a call small
# enough for the split decoder
CASES = [
    ("llama8b_t16k", 300, 256, None),
    ("glm4_9b_t32k", 300, 256, None),
    ("opt125m_t256", 256, 256, None),
    ("custom_1032", 260, 128, [(0, 2, 64), (2, 4, 8)]),
]


def _case(name, T, specs):
    if name == "custom_1032":
        rng = np.random.default_rng(5)
        L, H, D = 4, 8, 129
        x = rng.standard_normal((L, 2, T, H * D)).astype(np.float32)
        bits = (x.view(np.uint32) >> 16).astype(np.uint16)
        return bits, H, D, specs, specs
    p = synthetic.WORKLOADS[name]
    k, v = synthetic.workload_specs(name)
    return synthetic.generate(name, num_tokens=T), p["H"], p["D"], k, v


@pytest.fixture(scope="module", params=["CG_TEST_TARGET_MISS", "CG_TEST_EXACT_PATHS"])
def variant(request):
    return build.build_test_variant("test_" + request.param.lower(), [request.param])


@pytest.mark.parametrize("name,T,chunk,specs", CASES, ids=[c[0] for c in CASES])
def test_forced_exact_paths_match_the_oracle(orc, variant, name, T, chunk, specs):
    bits, H, D, k, v = _case(name, T, specs)
    L, _, T, C = bits.shape
    ref = orc.encode(bits, chunk, k, v)
    want = orc.decode(ref, L, T, C, chunk, k, v)
    with cg.use_library(variant):
        codec = cg.Codec(L, T, H, D, chunk, k, v)
        enc = codec.encode(_to_dev(bits, H, D))
        out = codec.decode(enc)
        torch.cuda.synchronize()
        assert enc.stream_bytes == ref["stream_bytes"]
        assert np.array_equal(enc.lengths.cpu().numpy(), ref["lengths"])
        assert np.array_equal(enc.cdf.cpu().numpy().view(np.uint16), ref["cdf"])
        assert np.array_equal(enc.bytestream[:enc.stream_bytes].cpu().numpy(), ref["bytes"])
        assert np.array_equal(_bits(out).reshape(L, 2, T, C), want)
        del codec, enc, out


def test_a_decoder_wait_that_runs_out_is_reported(orc):
    """The decoder's wait for its table copy is bounded: in a build whose
    barrier expects 16 bytes more than the copy brings, the wait runs out,
    the call reports CG_ERR_TIMEOUT and returns, and the context stays
    usable (the product library then decodes the same streams exactly)."""
    name, T = "mistral7b_t1k", 300
    bits, H, D, k, v = _case(name, T, None)
    L, _, T, C = bits.shape
    codec = cg.Codec(L, T, H, D, 256, k, v)
    enc = codec.encode(_to_dev(bits, H, D))
    lib = build.build_test_variant("test_cg_test_wait_timeout", ["CG_TEST_WAIT_TIMEOUT"])
    with cg.use_library(lib):
        with pytest.raises(cg.CacheGenError) as e:
            codec.decode(enc)
        assert e.value.status == cg.CG_ERR_TIMEOUT
    torch.cuda.synchronize()
    ref = orc.encode(bits, 256, k, v)
    out = codec.decode(enc)
    assert np.array_equal(_bits(out).reshape(L, 2, T, C), orc.decode(ref, L, T, C, 256, k, v))
