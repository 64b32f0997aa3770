"""Host-side logic of bench.py: the recorded DRAM traffic is reported only while the
kernel's sources hash to the value recorded beside it, and the byte counts."""
import bench


def test_recorded_traffic_follows_the_source_hash(tmp_path, monkeypatch):
    h = bench.kernel_source_hash("adaln_block_kernel")
    record = tmp_path / "dram_traffic.txt"
    record.write_text(f"# comment line\nadaln_block_kernel {h} 1106380800\n")
    assert bench.recorded_traffic("adaln_block_kernel", str(record)) == 1106380800
    assert bench.recorded_traffic("swiglu_kernel", str(record)) is None
    monkeypatch.setattr(bench, "kernel_source_hash", lambda kernel: "0" * 16)
    assert bench.recorded_traffic("adaln_block_kernel", str(record)) is None
    assert bench.recorded_traffic("adaln_block_kernel", str(tmp_path / "missing.txt")) is None


def test_source_hash_covers_the_kernel_and_the_shared_header():
    assert bench.KERNEL_SOURCES["adaln_block_kernel"] == ("adaln.cu", "h3q_device.cuh")
    assert len(bench.kernel_source_hash("swiglu_kernel")) == 16
    assert bench.kernel_source_hash("swiglu_kernel") != bench.kernel_source_hash("quantize_kernel")


def test_algorithmic_bytes():
    # x read once, codes and swizzled scales (padded to 128 rows) written once, tables once
    assert bench.adaln_bytes(65280, 7168, 32) == 1_199_994_884
    assert bench.quantize_bytes(8192, 7168) == 150_470_660
    assert bench.swiglu_bytes(65280, 18944) == 5_642_280_964


def test_recorded_instruction_counts_follow_the_source_hash(tmp_path, monkeypatch):
    h = bench.kernel_source_hash("swiglu_kernel")
    record = tmp_path / "inst_per_element.txt"
    record.write_text(f"# comment\nswiglu_kernel {h} 20.037\n")
    assert bench.recorded_value("swiglu_kernel", str(record)) == 20.037
    monkeypatch.setattr(bench, "kernel_source_hash", lambda kernel: "f" * 16)
    assert bench.recorded_value("swiglu_kernel", str(record)) is None


def test_qkv_bytes():
    # q, k, v read and written, three biases, cos and sin once
    assert bench.qkv_bytes(65280, 56, 128, 64) == 3 * 2 * 65280 * 7168 * 2 + 3 * 7168 * 2 + 2 * 65280 * 64 * 2


def test_link_bound():
    link = {"h2d_gbs": 200.0, "d2h_gbs": 100.0, "both_gbs_each": 50.0}
    # 1 GB in, 0.5 GB out: 0.5 GB each way at 50 GB/s (10 ms), then 0.5 GB in at 200 GB/s (2.5 ms)
    assert abs(bench.link_bound_ms(10 ** 9, 5 * 10 ** 8, link) - 12.5) < 1e-9
    # the larger direction out: its own one-way rate for the rest
    assert abs(bench.link_bound_ms(5 * 10 ** 8, 10 ** 9, link) - 15.0) < 1e-9


def test_source_hash_ignores_comments_and_whitespace():
    code = "int f(int a) {\n  return a + 1;  // one\n}\n"
    assert bench._code_only(code) == bench._code_only("/* header */\nint f(int a) { return a + 1; }")
    assert bench._code_only(code) != bench._code_only("int f(int a) { return a + 2; }")


def test_producer_oracle_timings_run_on_the_host():
    for kind in ("swiglu", "swiglu_packed", "quantize", "residual", "qkv"):
        r = bench.producer_oracle(kind, seconds=0.01, rows=8)
        assert r["gbs"] > 0 and r["kind"] == "oracle" and r["cores"] >= 1
