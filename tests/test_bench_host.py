"""Host-side arithmetic of the bench: the transfer-time model and the
relative reconstruction error, on CPU."""
import os
import sys

import pytest

torch = pytest.importorskip("torch")
sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402


def test_transfer_model_closed_forms():
    m = bench.transfer_model(10 ** 9, {"cachegen": 2 * 10 ** 8, "int8": 5 * 10 ** 8},
                             {"cachegen": 3.0, "int8": 1.0})
    assert m["bandwidth_mbps"] == [100, 500, 1000]
    # 1 GB = 8 Gbit: 80 s, 16 s, 8 s
    assert m["raw_s"] == [80.0, 16.0, 8.0]
    # 0.2 GB plus 3 ms of decode
    assert m["cachegen_s"] == [16.003, 3.203, 1.603]
    assert m["int8_s"] == [40.001, 8.001, 4.001]


def test_rel_rmse():
    x = torch.ones((2, 2, 3, 4), dtype=torch.bfloat16)
    assert bench.rel_rmse(x, x) == 0.0
    y = x * 1.5
    assert abs(bench.rel_rmse(x, y) - 0.5) < 1e-12
    assert bench.rel_rmse(torch.zeros_like(x), y) == 0.0


def test_sweep_settings_are_valid_spec_lists(orc):
    for L in (6, 12, 32, 40):
        seen = set()
        for label, k, v in bench.sweep_settings(L):
            assert label not in seen
            seen.add(label)
            orc.layer_bins(L, k)   # raises on lists that do not tile [0, L)
            orc.layer_bins(L, v)
        assert "preset" in seen and "uniform16" in seen


def test_issue_ceiling_arithmetic():
    r = bench.issue_ceiling("no_such_kernel", "llama8b_t16k", 2.0, 152, 2070.0)
    assert r["bound"] == "alu" and r["achieved"] is None and r["frac"] is None
    assert r["peak"] == 152 * 4 * 2070e6
    r = bench.issue_ceiling("no_such_kernel", "llama8b_t16k", 2.0, 100, None)
    assert r["peak"] == 100 * 4 * bench.NOMINAL_SM_MHZ * 1e6


def test_cpu_baseline_small_sample(orc):
    c = bench.cpu_baseline("opt125m_t256", 32)
    assert c["kind"] == "oracle" and c["value"] > 0 and c["cores"] >= 1
    assert c["single_core"]["value"] > 0


def test_code_hash_ignores_comments_only():
    a = "int f(int x) { return x + 1; } // one\n/* two */\n"
    b = "int f(int x)\n{\n    return x + 1;  /* changed */\n}\n"
    c = "int f(int x) { return x + 2; }"
    assert bench.code_hash(a) == bench.code_hash(b)
    assert bench.code_hash(a) != bench.code_hash(c)



def test_recorded_counters_belong_to_the_current_kernel_source():
    """profiles/traffic.json holds one-pass ncu counters of whole calls; the
    bench reports them only while they match the kernel source they were
    taken on. Every entry must carry the current source's hash, i.e. the
    counters were taken again after the last change to the kernels."""
    import json
    with open(os.path.join(os.path.dirname(bench.KERNEL_SOURCE), "..", "..", "profiles",
                           "traffic.json")) as f:
        d = json.load(f)
    sha = bench.kernel_source_hash()
    entries = [(k, w, e) for k, v in d.items() if not k.startswith("_") for w, e in v.items()]
    assert entries
    for kernel, workload, e in entries:
        assert e["source_sha"] == sha, (kernel, workload)
        assert e["dram_bytes_per_launch"] > 0 and e["warp_instructions_per_launch"] > 0
    for workload in ("llama8b_t16k", "glm4_9b_t32k"):
        for kernel in ("k_encode_tiles", "k_decode_tiles"):
            assert bench.recorded_counter(kernel, workload) == d[kernel][workload][
                "dram_bytes_per_launch"]
