"""The in-tree build's cache: a library is compiled once per source digest
and set of test macros, and reused while neither changes. The compiler is
replaced by a stub that writes a placeholder file, so this runs on CPU
without nvcc."""
import os

from kv_cache_compression_03_gb300 import build


def _stub(calls):
    def compile_(out_dir, lib, defines=()):
        calls.append((os.path.basename(out_dir), tuple(defines)))
        with open(lib, "w") as f:
            f.write("stub")
        return ""
    return compile_


def test_a_build_is_reused_until_its_sources_or_macros_change(tmp_path, monkeypatch):
    calls = []
    monkeypatch.setattr(build, "_compile", _stub(calls))
    digest = ["aaaa"]
    monkeypatch.setattr(build, "_digest", lambda: digest[0])
    out = str(tmp_path / "lib")

    lib = build._build_into(out)
    assert os.path.exists(lib) and len(calls) == 1
    build._build_into(out)                      # same sources: reused
    assert len(calls) == 1
    build._build_into(out, ("CG_TEST_X",))      # a macro set is another build
    assert len(calls) == 2
    build._build_into(out, ("CG_TEST_X",))
    assert len(calls) == 2
    digest[0] = "bbbb"                          # sources changed: rebuilt
    build._build_into(out, ("CG_TEST_X",))
    assert len(calls) == 3
    build._build_into(out, force=True)          # forced
    assert len(calls) == 4


def test_test_variants_live_beside_the_product_library(tmp_path, monkeypatch):
    calls = []
    monkeypatch.setattr(build, "_compile", _stub(calls))
    monkeypatch.setattr(build, "OUT_DIR", str(tmp_path))
    lib = build.build_test_variant("test_cg_test_x", ["CG_TEST_X"])
    assert lib == os.path.join(str(tmp_path), "test_cg_test_x", "libcachegen.so")
    assert calls == [("test_cg_test_x", ("CG_TEST_X",))]
