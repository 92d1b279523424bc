"""Host logic of bench.py that needs no GPU: the algorithmic byte count of a verify step and the
DRAM-traffic figure it reports only while the persistent kernel's sources match the capture."""
import pytest

import bench
import fixtures as FX


def test_verify_bytes_8b():
    """Every weight once (15.009 GB at the 8B shape), the KV prefix once per layer (131,072 B per
    token: 32 layers x K and V x 8 KV heads x 128 dims x 2 bytes) and the new K/V rows."""
    m = FX.WORKLOADS["8b_eagle2"].model
    weights = bench.verify_bytes(m, 1, 0, 0)
    assert abs(weights - 15.009e9) < 0.001e9
    per_token = bench.verify_bytes(m, 1, 1, 0) - weights
    assert per_token == 32 * 2 * 8 * 128 * 2
    assert bench.verify_bytes(m, 1, 0, 61) - weights == 61 * per_token
    assert bench.verify_bytes(m, 4, 1, 0) - weights == 4 * per_token


def test_traffic_follows_the_source_hash(tmp_path, monkeypatch):
    h = bench.kernel_source_hash()
    f = tmp_path / "traffic.txt"
    f.write_text("# comment\nkernel: stack_tc_kernel\ndram_bytes_read_per_launch: 100\n"
                 f"dram_bytes_write_per_launch: 23\nsource_sha256_16: {h}\n")
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(f))
    assert bench.captured_traffic() == 123
    f.write_text(f.read_text().replace(h, "0" * 16))  # the kernel changed since the capture
    assert bench.captured_traffic() is None
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(tmp_path / "missing.txt"))
    assert bench.captured_traffic() is None


def test_committed_traffic_is_close_to_algorithmic():
    """The committed capture, while it is of these sources, is close to the algorithmic bytes
    (no weight read twice)."""
    t = bench.captured_traffic()
    if t is None:
        pytest.skip("the committed DRAM capture predates the current kernel sources")
    m = FX.WORKLOADS["8b_eagle2"].model
    assert 1.0 <= t / bench.verify_bytes(m, 1, 1040, 61) < 1.05
