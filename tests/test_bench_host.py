"""Host-side pieces of bench.py (no GPU): it imports, its argument parser
runs, and its stored traffic record and work formulas are self-consistent."""
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_traffic_record_is_consistent():
    rec = bench.TRAFFIC_RECORD
    assert len(rec["source_sha1"]) == 40
    per = rec["per_launch_gb"]
    assert abs(rec["bytes_per_step"] / 1e9 - (per["fwd_saved"] + per["dh"])) < 0.02
    sha = bench.kernel_source_sha1()
    assert len(sha) == 40 and all(c in "0123456789abcdef" for c in sha)


def test_algorithmic_bytes_of_the_step():
    # forward: h + W read, partials + target logits + terms written; the
    # conversion pass: terms read, dZ written, partials read; dh GEMM: dZ + W
    # read, dh written (71.48 GB at T = 65536, H = 4096, V = 128256)
    assert bench.algorithmic_bytes_per_step(65536, 4096, 128256) == 71480639488


def test_cli_parses():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--help"],
                       capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and "--steps" in r.stdout
