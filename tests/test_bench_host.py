"""Host-side logic of bench.py: the recorded DRAM traffic is reported only while the
kernel's sources hash to the value recorded beside it, and the byte counts."""
import bench


def test_recorded_traffic_follows_the_source_hash(monkeypatch):
    value = bench.recorded_traffic("adaln_block_kernel")
    assert value is not None and value > 0
    # ~ the algorithmic bytes of the 65,280 x 7,168 workload (reads once, writes partly in L2)
    assert 0.8 * bench.adaln_bytes(65280, 7168, 32) < value < 1.2 * bench.adaln_bytes(65280, 7168, 32)
    monkeypatch.setattr(bench, "kernel_source_hash", lambda kernel: "0" * 16)
    assert bench.recorded_traffic("adaln_block_kernel") is None
    assert bench.recorded_traffic("no_such_kernel") is None


def test_algorithmic_bytes():
    # x read once, codes and swizzled scales (padded to 128 rows) written once, tables once
    assert bench.adaln_bytes(65280, 7168, 32) == 1_199_994_884
    assert bench.quantize_bytes(8192, 7168) == 150_470_660
    assert bench.swiglu_bytes(65280, 18944) == 5_642_280_964
