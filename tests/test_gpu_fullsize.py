"""Parity at the full workload sizes, in the bench's launch configuration:
the whole blob is encoded and decoded on the GPU, and sampled tiles are
checked against the oracle (which encodes only those tiles): scales, CDF
blocks, stream lengths, stream bytes, and the decoded bf16 rows."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

from kv_cache_compression_03_gb300 import cachegen as cg  # noqa: E402
from kv_cache_compression_03_gb300 import synthetic  # noqa: E402


@pytest.mark.parametrize("name", ["llama8b_t16k", "glm4_9b_t32k"])
def test_full_size_sampled_tiles(orc, name):
    p = synthetic.WORKLOADS[name]
    k, v = synthetic.workload_specs(name)
    L, T, H, D = p["L"], p["T"], p["H"], p["D"]
    C = H * D
    ch = p["chunk_tokens"][0]
    bits = synthetic.generate(name)
    codec = cg.Codec(L, T, H, D, ch, k, v)
    kv = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).reshape(L, 2, T, H, D).cuda()
    enc = codec.encode(kv)
    out = codec.decode(enc)
    torch.cuda.synchronize()

    kb, vb = orc.layer_bins(L, k), orc.layer_bins(L, v)
    gs, gc = orc.groups(T, ch)
    ng = len(gs)
    ntiles = ng * 2 * L
    lengths = enc.lengths.cpu().numpy().astype(np.int64)
    assert lengths.min() >= 1
    offsets = np.concatenate([[0], np.cumsum(lengths)])
    assert offsets[-1] == enc.stream_bytes
    # every CDF row of the whole table is a valid CDF
    cdf = enc.cdf.cpu().numpy().view(np.uint16)
    rng = np.random.default_rng(17)
    pick = sorted(set([0, ntiles - 1, L - 1, L, 2 * L * (ng // 2) + 3] +
                      rng.integers(0, ntiles, 6).tolist()))
    got = orc.encode_tiles(bits, ch, k, v, pick)
    per_group = sum(C * (int(b) + 1) for b in list(kb) + list(vb))
    amax = enc.amax.cpu().numpy()
    out_bits = out.view(torch.int16).cpu().numpy().view(np.uint16).reshape(L, 2, T, C)
    stream = enc.bytestream[:enc.stream_bytes].cpu().numpy()
    for t in got:
        ti = t["tile"]
        g, kvs, l = ti // (2 * L), (ti // L) % 2, ti % L
        N = int((kb, vb)[kvs][l])
        n = int(gc[g])
        first = 2 * L * int(gs[g]) + (kvs * L + l) * n
        off = g * per_group + sum(C * (int(b) + 1) for b in
                                  (list(kb) + list(vb))[:kvs * L + l])
        assert np.array_equal(cdf[off:off + C * (N + 1)], t["cdf"])
        assert np.array_equal(lengths[first:first + n], t["lengths"])
        assert np.array_equal(amax[kvs, l, gs[g]:gs[g] + n], t["amax"])
        b0 = offsets[first]
        assert np.array_equal(stream[b0:b0 + int(t["lengths"].sum())], t["bytes"])
        rows = t["cdf"].reshape(C, N + 1).astype(np.uint32)
        rows[:, N] = 65536
        bins = N
        pos = 0
        for i in range(n):
            ln = int(t["lengths"][i])
            q = orc.wnc_decode(t["bytes"][pos:pos + ln].tobytes(), C, rows)
            pos += ln
            want = orc.dequant_row(q, bins, float(t["amax"][i]))
            assert np.array_equal(out_bits[l, kvs, gs[g] + i], want)
    # the reconstruction bound holds everywhere (sampled rows of every layer)
    x = kv.reshape(L, 2, T, C)[:, :, ::97].float().double()
    y = out.reshape(L, 2, T, C)[:, :, ::97].float().double()
    a = enc.amax.permute(1, 0, 2)[:, :, ::97].double()[..., None]
    M = torch.tensor([[b // 2 - 1 for b in (kb[l], vb[l])] for l in range(L)],
                     dtype=torch.float64, device=a.device)[:, :, None, None]
    bound = 0.5 * a / M * (1 + 2.0 ** -20) + y.abs() * 2.0 ** -8
    assert bool(((x - y).abs() <= bound).all())
