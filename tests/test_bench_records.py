"""The benchmark's traffic records on CPU: a record of DRAM bytes per launch is reported only while
the kernel's source and every header it includes are the ones it was captured with. Checked on a
copy of the source tree, so that edits can be made without touching the repository."""
import json
import os
import shutil
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


@pytest.fixture
def tree(tmp_path, monkeypatch):
    """A copy of the kernel sources, the public header and the profiles, with bench pointed at it."""
    for d in ("include", "profiles"):
        shutil.copytree(os.path.join(ROOT, d), tmp_path / d)
    shutil.copytree(os.path.join(ROOT, "bit_quantized_routed_gb300", "csrc"),
                    tmp_path / "bit_quantized_routed_gb300" / "csrc")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    return tmp_path


def _names(files):
    return sorted(os.path.basename(f) for f in files)


def test_closure_follows_nested_includes_only(tree):
    # gemm_tc.cu includes common.cuh and ptx.cuh; common.cuh includes internal.h, which includes
    # the public header; the single-token kernel's helpers are not in it
    got = _names(bench._include_closure(("gemm_tc.cu",)))
    assert got == ["common.cuh", "ds4moe.h", "gemm_tc.cu", "internal.h", "ptx.cuh"]
    got = _names(bench._include_closure(("decode_step.cu",)))
    assert "step_common.cuh" in got and "ds4moe.h" in got and "gemm_tc.cu" not in got


def _append(path, text):
    with open(path, "a") as f:
        f.write(text)


def test_hash_changes_with_the_closure_and_nothing_else(tree):
    csrc = tree / "bit_quantized_routed_gb300" / "csrc"
    g0, d0 = bench.src_sha("gemm_tc.cu"), bench.src_sha("decode_step.cu")
    _append(csrc / "step_common.cuh", "\n// an edit\n")  # in the single-token kernel's closure only
    assert bench.src_sha("gemm_tc.cu") == g0
    d1 = bench.src_sha("decode_step.cu")
    assert d1 != d0
    _append(tree / "include" / "ds4moe.h", "\n/* an edit */\n")  # in every kernel's closure
    assert bench.src_sha("gemm_tc.cu") != g0
    assert bench.src_sha("decode_step.cu") != d1


def test_record_is_reported_only_while_its_source_is_unchanged(tree):
    path = tree / "profiles" / "traffic.json"
    db = json.load(open(path))
    key = "gemm_kernel<UP>@prefill_t8192_d7168"
    db[key] = {"src_sha": bench.src_sha("gemm_tc.cu"), "bytes_per_launch": 123456}
    json.dump(db, open(path, "w"))
    assert bench.ncu_traffic("up_gemm", "prefill_t8192_d7168") == 123456
    _append(tree / "bit_quantized_routed_gb300" / "csrc" / "gemm_tc.cu", "\n// an edit\n")
    assert bench.ncu_traffic("up_gemm", "prefill_t8192_d7168") is None
