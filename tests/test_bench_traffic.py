"""bench.py's traffic check reads a committed ncu summary only while every
source file it lists still has the SHA-256 it was captured on (host logic,
no GPU)."""
import hashlib
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _tree(tmp_path, src_text, listed_sha=None):
    pkg = tmp_path / "block_diffusion_speculative_02_gb300" / "csrc"
    pkg.mkdir(parents=True)
    (pkg / "k.cu").write_text(src_text)
    (pkg / "c.cuh").write_text("// common\n")
    sha_k = listed_sha or hashlib.sha256(src_text.encode()).hexdigest()[:16]
    sha_c = hashlib.sha256(b"// common\n").hexdigest()[:16]
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "k.md").write_text(
        "# a kernel\n\n"
        f"source_sha256: csrc/k.cu={sha_k} csrc/c.cuh={sha_c}\n"
        "traffic_bytes_per_launch: 1010\n"
        "algorithmic_bytes_per_launch: 1000\n"
        "traffic_bytes_per_launch[B]: 2200\n"
        "algorithmic_bytes_per_launch[B]: 2000\n")


def test_matching_sources_give_the_ratio(tmp_path, monkeypatch):
    _tree(tmp_path, "__global__ void k() {}\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    t = bench.profiled_traffic("k.md")
    assert t["traffic"] == 1010 and t["algorithmic"] == 1000
    assert abs(t["ratio"] - 1.01) < 1e-12
    tb = bench.profiled_traffic("k.md", "B")
    assert tb["traffic"] == 2200 and abs(tb["ratio"] - 1.1) < 1e-12
    assert bench.profiled_traffic("k.md", "C") is None           # no such entry


def test_a_changed_source_drops_the_figure(tmp_path, monkeypatch):
    _tree(tmp_path, "__global__ void k() {}\n", listed_sha="0123456789abcdef")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profiled_traffic("k.md") is None
    assert bench.profiled_traffic("missing.md") is None


def test_committed_summaries_parse():
    """Every committed summary that lists source hashes names files that exist
    and carries well-formed traffic lines (whether the hashes are current is
    what the bench reports, not a test failure)."""
    prof = os.path.join(ROOT, "profiles")
    for name in sorted(os.listdir(prof)):
        lines = open(os.path.join(prof, name), encoding="utf-8").read().splitlines()
        srcs = [l for l in lines if l.startswith("source_sha256:")]
        if not srcs:
            continue
        assert len(srcs) == 1, name
        for pair in srcs[0].split(":", 1)[1].split():
            rel, sha = pair.split("=")
            assert os.path.exists(os.path.join(ROOT, "block_diffusion_speculative_02_gb300", rel)), (name, rel)
            assert len(sha) == 16 and int(sha, 16) >= 0, (name, pair)
        for l in lines:
            if l.startswith(("traffic_bytes_per_launch", "algorithmic_bytes_per_launch")):
                assert float(l.split(":", 1)[1]) > 0, (name, l)
