"""Static checks of the repository layout (CPU): the product package never
imports the oracle, and no committed source reads the working folder."""
import os
import re
import subprocess

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "trainable_sparse_attention_gb300")


def _tracked(suffixes):
    out = subprocess.run(["git", "ls-files"], cwd=ROOT, capture_output=True, text=True)
    if out.returncode != 0:  # not a git checkout: walk the tree instead
        files = []
        for d, _, fs in os.walk(ROOT):
            if "/_work" in d or "/.git" in d:
                continue
            files += [os.path.relpath(os.path.join(d, f), ROOT) for f in fs]
    else:
        files = out.stdout.split()
    return [f for f in files if f.endswith(suffixes)]


def test_product_package_never_imports_the_oracle():
    pat = re.compile(r"^\s*(from\s+oracle\b|import\s+oracle\b)|\boracle\.", re.M)
    for d, _, fs in os.walk(PKG):
        for f in fs:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                src = open(os.path.join(d, f), encoding="utf-8").read()
                assert not pat.search(src), f"{f} refers to the oracle"


def test_oracle_is_imported_only_by_tests_smoke_and_the_bench_baselines():
    allowed = {"__graft_entry__.py", "bench.py"}
    for f in _tracked((".py",)):
        if f.startswith(("tests/", "oracle/")) or f in allowed:
            continue
        src = open(os.path.join(ROOT, f), encoding="utf-8").read()
        assert not re.search(r"^\s*(from\s+oracle\b|import\s+oracle\b)", src, re.M), f


def test_no_committed_file_reads_the_working_folder():
    marker = "_" + "work" + "/"  # built here so that this file does not match itself
    for f in _tracked((".py", ".cu", ".cuh", ".h", ".sh")):
        src = open(os.path.join(ROOT, f), encoding="utf-8").read()
        assert marker not in src, f


def test_every_kernel_launch_is_counted():
    """Each <<<...>>> statement of the library is followed by note_launch(), so the
    launch count (tsa_kernel_launches, the bench's gpu_launches) is exact."""
    csrc = os.path.join(PKG, "csrc")
    sites = 0
    for f in sorted(os.listdir(csrc)):
        if not f.endswith(".cu"):
            continue
        lines = open(os.path.join(csrc, f), encoding="utf-8").read().split("\n")
        for i, ln in enumerate(lines):
            if "<<<" in ln and not ln.lstrip().startswith("//"):
                sites += 1
                assert lines[i + 1].strip() == "note_launch();", f"{f}:{i + 1} launch not counted"
    assert sites >= 18
