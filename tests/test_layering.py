"""The product path and the oracle stay apart, and the product fails loudly
without its compiled library (no CPU fallback exists to fall back to)."""
from __future__ import annotations

import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "mxfp4_expert_ffn_gb300")


def _files(*patterns):
    out = []
    for p in patterns:
        out += glob.glob(os.path.join(ROOT, p), recursive=True)
    return sorted(out)


def test_package_never_imports_the_oracle():
    for f in _files("mxfp4_expert_ffn_gb300/**/*.py"):
        src = open(f).read()
        assert not re.search(r"^\s*(import|from)\s+oracle\b", src, re.M), f


def test_cuda_sources_and_oracle_share_no_code():
    for f in _files("mxfp4_expert_ffn_gb300/csrc/*", "include/*.h"):
        assert "oracle" not in "".join(re.findall(r'#include\s*[<"]([^>"]+)', open(f).read())), f
    inc = re.findall(r'#include\s*[<"]([^>"]+)', open(os.path.join(ROOT, "oracle", "oracle.c")).read())
    assert all("/" not in i and not i.endswith((".cuh", ".cu")) and i != "moe_ffn.h" for i in inc), inc


def test_oracle_is_used_only_by_tests_smoke_and_the_bench_baseline():
    rels = [os.path.relpath(f, ROOT) for f in _files("**/*.py")]
    users = [r for r in rels if not r.startswith(("_work/", "tests/", "oracle/", "baseline/"))
             and re.search(r"^\s*(import|from)\s+oracle\b", open(os.path.join(ROOT, r)).read(), re.M)]
    assert sorted(users) == ["__graft_entry__.py", "bench.py"]
    # in the bench, only the CPU baseline and the reference arm import it: inside
    # their own functions, or in the block the --no-cpu-baseline switch guards
    lines = open(os.path.join(ROOT, "bench.py")).read().splitlines()
    func = None
    for i, line in enumerate(lines):
        if line.startswith("def "):
            func = line[4:].split("(")[0]
        if re.match(r"^\s+import oracle\b", line):
            guarded = "no_cpu_baseline" in lines[i - 1]
            assert guarded or any(w in func for w in ("cpu", "reference", "oracle")), (i + 1, func)


def test_missing_library_raises_instead_of_falling_back(monkeypatch):
    import mxfp4_expert_ffn_gb300 as m
    monkeypatch.setattr(m, "_lib", None)
    monkeypatch.setattr(m, "LIB_PATH", os.path.join(ROOT, "no_such_dir", "libmoe_ffn.so"))
    with pytest.raises(RuntimeError, match="missing"):
        m.lib()
