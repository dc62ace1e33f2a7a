"""Host logic of the benchmark that needs no GPU: reading the committed ncu
summaries, and the summaries themselves (each names the command that made it)."""
from __future__ import annotations

import glob
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _write_profile(root, name, digest, extra=""):
    os.makedirs(os.path.join(root, "profiles"), exist_ok=True)
    with open(os.path.join(root, "profiles", name), "w") as f:
        f.write("# a summary\n\ntraffic_bytes_per_launch: 2532274800\n"
                f"source_digest: `{digest}`\n{extra}")


def test_stored_profile_needs_the_current_digest(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_digest", lambda k: "abc123")
    _write_profile(str(tmp_path), "prefix_tc_mixed_serving.md", "abc123",
                   "captured_algorithmic_bytes: 2505339904\ntensor_pipe_active_pct: 26.3\n")
    got = bench.stored_profile("prefix_tc", "mixed_serving")
    assert got == {"traffic": 2532274800, "tensor_pipe_active_pct": 26.3,
                   "captured_algorithmic_bytes": 2505339904}
    _write_profile(str(tmp_path), "prefix_tc_llama8b_gqa.md", "stale")
    assert bench.stored_profile("prefix_tc", "llama8b_gqa") == {}
    assert bench.stored_profile("prefix_tc", "no_such_workload") == {}


def test_committed_summaries_name_their_command_and_a_known_kernel():
    files = sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md")))
    assert files
    for path in files:
        text = open(path).read()
        assert "ncu " in text, f"{os.path.basename(path)} gives no ncu command"
        assert "--clock-control none" in text, os.path.basename(path)
        for line in text.splitlines():
            if line.startswith("source_digest:"):
                kernel = [k for k in bench.KERNEL_SOURCES if os.path.basename(path).startswith(k + "_")]
                assert kernel, f"{os.path.basename(path)}: digest for an unknown kernel"


def test_every_kernel_digest_reads_existing_sources():
    for k in bench.KERNEL_SOURCES:
        d = bench.kernel_digest(k)
        assert isinstance(d, str) and len(d) == 16
