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

