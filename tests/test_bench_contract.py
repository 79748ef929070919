"""The bench's JSON line: the keys and types the measurement contract asks
for. The reference arm (the CPU oracle) runs here; the codec arm needs a
GPU."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
BASE_KEYS = {"metric": str, "value": (int, float), "unit": str, "n_gpus": int, "steps": int,
             "warmup": int, "ms_per_step": (int, float), "higher_is_better": bool,
             "scaling": str, "dtype": str, "data": str, "config": dict, "e2e": dict,
             "cpu_baseline": dict}


def _run(args, timeout=600):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py")] + args, cwd=ROOT,
                       capture_output=True, text=True, timeout=timeout)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [x for x in r.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1, r.stdout
    return json.loads(lines[0])


def _check_base(d):
    for k, t in BASE_KEYS.items():
        assert k in d and isinstance(d[k], t), k
    assert d["config"]["workload"] == "llama8b_t16k"
    assert d["scaling"] == "weak" and d["higher_is_better"] is True
    assert d["vs_baseline"] is None
    for k in ("value", "unit", "h2d_bytes_per_step", "d2h_bytes_per_step"):
        assert k in d["e2e"]
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1


def test_reference_arm_line():
    d = _run(["--impl", "reference", "--steps", "1", "--warmup", "3", "--cpu-tokens", "16"])
    _check_base(d)
    assert d["impl"] == "reference" and d["e2e"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["gpu_launches"] == 0


def test_warmup_below_three_is_refused():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--warmup", "2"],
                       cwd=ROOT, capture_output=True, text=True, timeout=120)
    assert r.returncode != 0


@pytest.mark.gpu
def test_codec_arm_line():
    d = _run(["--steps", "3", "--warmup", "3", "--tokens", "1024", "--cpu-tokens", "64"])
    _check_base(d)
    assert "impl" not in d or d["impl"] != "reference"
    r = d["roofline"]
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and 0 < r["frac"] < 1.5
    assert abs(r["achieved"] / r["peak"] - r["frac"]) < 1e-3
    assert d["issue"]["bound"] == "alu"
    assert d["gpu_launches"] > 0 and d["clocks"] is not None
    assert d["e2e"]["h2d_bytes_per_step"] > 0 and d["e2e"]["d2h_bytes_per_step"] > 0
    b = d["baselines"]
    assert b["int8"]["compression_ratio"] == pytest.approx(2 * 1024 / 1028, rel=1e-3)
    assert b["naive"]["compression_ratio"] == 1.0
    assert set(b["transfer_model"]) >= {"bandwidth_mbps", "raw_s", "cachegen_s", "int8_s"}


def _lines(args, timeout=900):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py")] + args, cwd=ROOT,
                       capture_output=True, text=True, timeout=timeout)
    assert r.returncode == 0, r.stderr[-2000:]
    return [json.loads(x) for x in r.stdout.splitlines() if x.startswith("{")]


@pytest.mark.gpu
def test_bins_sweep_lines():
    rows = _lines(["--sweep-bins", "--tokens", "256", "--steps", "2", "--warmup", "3"])
    by = {r["setting"]: r for r in rows}
    assert {"preset", "uniform8", "uniform16", "uniform32", "uniform64"} <= set(by)
    # more bins: lower error, lower ratio
    assert by["uniform8"]["rel_rmse"] > by["uniform16"]["rel_rmse"] > by["uniform32"]["rel_rmse"]
    assert by["uniform8"]["compression_ratio"] > by["uniform16"]["compression_ratio"] \
        > by["uniform32"]["compression_ratio"]


@pytest.mark.gpu
def test_chunk_sweep_lines():
    rows = _lines(["--sweep-chunks", "--steps", "2", "--warmup", "3"])
    assert [r["chunk_tokens"] for r in rows] == [64, 128, 256, 768]
    for r in rows:
        assert abs(r["per_object_ratio"] - r["compression_ratio"]) < 1e-3 * r["compression_ratio"]
        assert r["objects"] == -(-768 // r["chunk_tokens"])
