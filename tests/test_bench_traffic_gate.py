"""The benchmark reports the ncu traffic of the statistics kernel only while the kernel source is
the one the capture was taken on: the summary records the source's hash, and any change to the
source turns the figure into null."""
import hashlib
import importlib.util
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_traffic_follows_the_source_hash(tmp_path, monkeypatch):
    bench = _bench()
    src = tmp_path / "kernel.cu"
    src.write_bytes(b"__global__ void k() {}\n")
    digest = hashlib.sha256(src.read_bytes()).hexdigest()[:16]
    (tmp_path / "summary.md").write_text(
        f"# a capture\n\ntraffic_bytes_per_launch: 123456\nkernel_source_sha256_16: {digest}\n")
    monkeypatch.setattr(bench, "PROFILE_DIR", str(tmp_path))
    monkeypatch.setattr(bench, "KERNEL_SOURCE", str(src))
    assert bench.recorded_traffic("summary.md")[0] == 123456
    src.write_bytes(b"__global__ void k() { }\n")          # the kernel changed since the capture
    assert bench.recorded_traffic("summary.md")[0] is None
    assert bench.recorded_traffic("absent.md")[0] is None
