"""Host-side rules of the benchmark that need no GPU."""
import hashlib
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_recorded_traffic_follows_the_kernel_source(tmp_path, monkeypatch):
    """DRAM traffic from a committed capture is reported only while the kernel
    source still hashes to the value recorded with it."""
    (tmp_path / "profiles").mkdir()
    src = tmp_path / "k.cu"
    src.write_bytes(b"kernel v1")
    sha = hashlib.sha256(b"kernel v1").hexdigest()[:16]
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(
        {"prefill": {"source_sha256_16": sha, "dram_bytes_per_launch": 3245473280}}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setitem(bench.KERNEL_SOURCES, "prefill", "k.cu")
    assert bench.recorded_traffic("prefill") == 3245473280
    src.write_bytes(b"kernel v2")
    assert bench.recorded_traffic("prefill") is None
    assert bench.recorded_traffic("decode") is None  # no entry


def test_workload_bytes_match_the_roofline_arithmetic():
    """Algorithmic bytes of the two headline workloads: 1540 B per (token, head)
    for prefill plus h0 and hT; the decode step reads and writes the state and
    moves its token vectors and outputs."""
    w = bench.PREFILL
    assert (w.B, w.T, w.H, w.dk, w.dv) == (8, 8192, 32, 128, 128)
    per_token_head = 4 * 128 * 2 + 128 * 4 + 4
    assert per_token_head == 1540
    state = w.B * w.H * 128 * 128 * 4
    assert bench.prefill_bytes(w) == w.B * w.T * w.H * per_token_head + 2 * state
    d = bench.DECODE
    assert bench.decode_bytes(d) > 2 * 256 * 32 * 128 * 128 * 4  # state in and out, plus vectors
