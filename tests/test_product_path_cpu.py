"""Host-side guarantees about the product path (no GPU needed).

* The package and its library never reach the oracle: no file of the
  package imports, opens or names it, so no result can come from a CPU path.
* A missing library is an error, never a fallback.
* The benchmark reports DRAM traffic only while the kernel source is the one
  the committed ncu record was taken from.
"""
import json
import os
import re

import pytest

import nvfp4_weight_only_w4a16_gb300 as P

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "nvfp4_weight_only_w4a16_gb300")


def _package_files():
    for d, _, files in os.walk(PKG):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                yield os.path.join(d, f)
    yield os.path.join(ROOT, "include", "nvfp4_moe.h")


def test_package_never_reaches_the_oracle():
    pat = re.compile(r"\boracle\b")
    for path in _package_files():
        text = open(path, encoding="utf-8").read()
        for ln, line in enumerate(text.splitlines(), 1):
            assert not pat.search(line), f"{os.path.relpath(path, ROOT)}:{ln}: {line.strip()}"


def test_missing_library_is_an_error(tmp_path):
    with pytest.raises(FileNotFoundError):
        P.load_library(str(tmp_path / "libnvfp4moe.so"))


def test_traffic_record_follows_the_kernel_code(tmp_path, monkeypatch):
    import bench
    src = tmp_path / "kernel.cu"
    src.write_text("// v1\n__global__ void k(int* p) { p[0] = 1; }\n")
    rec = tmp_path / "record.json"
    rec.write_text(json.dumps({"code_sha256": bench.code_fingerprint(src.read_text()), "dram_bytes_per_launch": 12345}))
    monkeypatch.setattr(bench, "PROFILE_TRAFFIC", str(rec))
    assert bench._traffic_for(str(src)) == 12345
    src.write_text("/* a new comment */\n__global__ void k(int* p) {\n  p[0] = 1;  // same code\n}\n")
    assert bench._traffic_for(str(src)) == 12345   # comments and layout do not matter
    src.write_text("__global__ void k(int* p) { p[0] = 2; }\n")
    assert bench._traffic_for(str(src)) is None    # the code changed since the capture


def test_committed_traffic_record_is_consistent():
    import bench
    if not os.path.exists(bench.PROFILE_TRAFFIC):
        pytest.skip("no committed ncu traffic record for the bench's decode kernel: the bench reports traffic = null")
    rec = json.load(open(bench.PROFILE_TRAFFIC))
    assert rec["dram_bytes_per_launch"] == rec["dram_bytes_read_per_launch"] + rec["dram_bytes_write_per_launch"]
    src = os.path.join(ROOT, rec["source_file"])
    if bench.code_fingerprint(open(src, encoding="utf-8").read()) != rec["code_sha256"]:
        pytest.skip("the decode kernel's code changed since the committed ncu capture: the bench reports traffic = null")
