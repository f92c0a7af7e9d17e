"""bench.py reports a launch's DRAM traffic scaled from a stream's ncu
capture, and only while the device sources it was captured on are
unchanged (CPU)."""
import bench


def test_traffic_scales_with_descriptors(monkeypatch):
    monkeypatch.setattr(bench, "sources_digest", lambda: bench.TRAFFIC["c2"]["sources"])
    t = bench.TRAFFIC["c2"]
    assert bench.launch_traffic("c2", t["descs"]) == t["bytes"]
    assert bench.launch_traffic("c2", 10 * t["descs"]) == 10 * t["bytes"]
    assert bench.launch_traffic("no-such-stream", 100) is None


def test_traffic_withheld_once_the_kernel_changed(monkeypatch):
    monkeypatch.setattr(bench, "sources_digest", lambda: "0" * 16)
    for w in bench.TRAFFIC:
        assert bench.launch_traffic(w, 1000) is None


def test_digest_covers_the_device_sources():
    d = bench.sources_digest()
    assert len(d) == 16 and int(d, 16) >= 0
    assert all(f.endswith((".cu", ".h")) for f in bench.TRAFFIC_SOURCES)
