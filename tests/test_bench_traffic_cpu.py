"""bench.py reports the backward kernel's DRAM traffic from the committed ncu
summary only while the kernel sources are the ones that were profiled."""
import hashlib
import os
import shutil
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _tree(tmp_path, body_lines, sources):
    os.makedirs(tmp_path / "profiles")
    csrc = tmp_path / "packed_sequence_block_gb300" / "csrc"
    os.makedirs(csrc)
    for name, text in sources.items():
        (csrc / name).write_text(text)
    (tmp_path / "profiles" / "bd_bwd_kernel_lognormal8k.md").write_text("\n".join(body_lines) + "\n")
    return tmp_path


def _sha(text):
    return hashlib.sha256(text.encode()).hexdigest()


def test_traffic_follows_the_profiled_sources(tmp_path, monkeypatch):
    src = {"bd_bwd.cu": "kernel v1\n", "bd_ptx.cuh": "helpers v1\n"}
    root = _tree(tmp_path, ["    traffic_bytes_per_launch: 123456",
                            f"    source_sha256: bd_bwd.cu {_sha(src['bd_bwd.cu'])}",
                            f"    source_sha256: bd_ptx.cuh {_sha(src['bd_ptx.cuh'])}"], src)
    monkeypatch.setattr(bench, "ROOT", str(root))
    traffic, why = bench.profiled_traffic("lognormal8k", 0)
    assert traffic == 123456 and "ncu" in why
    # another workload or seed was never captured
    assert bench.profiled_traffic("lognormal8k", 1)[0] is None
    assert bench.profiled_traffic("shortdocs", 0)[0] is None
    # any change to a profiled source voids the figure
    (root / "packed_sequence_block_gb300" / "csrc" / "bd_ptx.cuh").write_text("helpers v2\n")
    traffic, why = bench.profiled_traffic("lognormal8k", 0)
    assert traffic is None and "bd_ptx.cuh changed" in why


def test_traffic_needs_both_the_figure_and_the_hashes(tmp_path, monkeypatch):
    src = {"bd_bwd.cu": "kernel v1\n"}
    root = _tree(tmp_path, ["    traffic_bytes_per_launch: 99"], src)
    monkeypatch.setattr(bench, "ROOT", str(root))
    assert bench.profiled_traffic("lognormal8k", 0)[0] is None
    shutil.rmtree(root / "profiles")
    assert bench.profiled_traffic("lognormal8k", 0) == (None, "no capture")


def test_committed_summary_parses():
    """The committed summary carries a figure and hashes for files that exist."""
    lines = open(os.path.join(ROOT, "profiles", "bd_bwd_kernel_lognormal8k.md")).read().splitlines()
    figures = [ln for ln in lines if ln.strip().startswith("traffic_bytes_per_launch:")]
    hashes = [ln.split(":", 1)[1].split() for ln in lines if ln.strip().startswith("source_sha256:")]
    assert len(figures) == 1 and int(figures[0].split(":", 1)[1]) > 0
    assert hashes
    for name, digest in hashes:
        assert os.path.exists(os.path.join(ROOT, "packed_sequence_block_gb300", "csrc", name))
        assert len(digest) == 64
