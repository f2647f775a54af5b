"""bench.py reports the backward kernel's DRAM traffic from the committed ncu
figures (a JSON file beside the prose summary) only while the kernel sources
are the ones that were profiled."""
import hashlib
import json
import os
import shutil
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

FIG = "bd_bwd_kernel_lognormal8k.json"


def _tree(tmp_path, fig, sources):
    os.makedirs(tmp_path / "profiles")
    csrc = tmp_path / "packed_sequence_block_gb300" / "csrc"
    os.makedirs(csrc)
    for name, text in sources.items():
        (csrc / name).write_text(text)
    (tmp_path / "profiles" / FIG).write_text(json.dumps(fig))
    return tmp_path


def _sha(text):
    return hashlib.sha256(text.encode()).hexdigest()


def test_traffic_follows_the_profiled_sources(tmp_path, monkeypatch):
    src = {"bd_bwd.cu": "kernel v1\n", "bd_ptx.cuh": "helpers v1\n"}
    fig = {"workload": "lognormal8k", "seed": 0, "traffic_bytes_per_launch": 123456,
           "source_sha256": {n: _sha(t) for n, t in src.items()}}
    root = _tree(tmp_path, fig, src)
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
    root = _tree(tmp_path, {"workload": "lognormal8k", "seed": 0,
                            "traffic_bytes_per_launch": 99}, src)
    monkeypatch.setattr(bench, "ROOT", str(root))
    assert bench.profiled_traffic("lognormal8k", 0)[0] is None
    shutil.rmtree(root / "profiles")
    assert bench.profiled_traffic("lognormal8k", 0) == (None, "no capture")


def test_committed_figures_parse():
    """The committed figures carry a traffic number and hashes of files that exist."""
    with open(os.path.join(ROOT, "profiles", FIG)) as f:
        fig = json.load(f)
    assert isinstance(fig["traffic_bytes_per_launch"], int) and fig["traffic_bytes_per_launch"] > 0
    assert fig["source_sha256"]
    for name, digest in fig["source_sha256"].items():
        assert os.path.exists(os.path.join(ROOT, "packed_sequence_block_gb300", "csrc", name))
        assert len(digest) == 64
