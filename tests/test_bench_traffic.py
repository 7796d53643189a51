"""The bench's ncu traffic figures are used only while they describe the
kernels as they are: an entry of profiles/traffic.txt lists the hash of every
source file its kernel is built from, and a figure whose sources changed
since the capture reads as null."""
import os
import shutil
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_a_changed_source_turns_the_figure_null(tmp_path, monkeypatch):
    # a copy of the tree's sources and traffic file in which one header differs
    root = tmp_path / "repo"
    shutil.copytree(os.path.join(ROOT, "paged_kv_cache_224_gb300", "csrc"),
                    root / "paged_kv_cache_224_gb300" / "csrc")
    shutil.copytree(os.path.join(ROOT, "profiles"), root / "profiles")
    monkeypatch.setattr(bench, "ROOT", str(root))
    # an entry keyed by the copy's own hashes is found ...
    h = ",".join(bench.source_hash(f) for f in bench.PREFILL_SOURCES)
    with open(root / "profiles" / "traffic.txt", "a") as f:
        f.write(f"probe_kernel {h} 12345\n")
    assert bench.load_traffic("probe_kernel", bench.PREFILL_SOURCES) == 12345.0
    hdr = root / "paged_kv_cache_224_gb300" / "csrc" / "pa_device.cuh"
    hdr.write_text(hdr.read_text() + "\n// changed\n")
    # ... and turns null once one of its sources changes
    assert bench.load_traffic("probe_kernel", bench.PREFILL_SOURCES) is None
    # an unknown kernel key has no figure
    assert bench.load_traffic("no_such_kernel", bench.DECODE_SOURCES) is None
