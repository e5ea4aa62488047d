"""Host-side helpers of bench.py (no GPU): the recorded-traffic lookup that
ties a committed ncu figure to the kernel source it was captured on, and the
CPU description that goes beside the CPU baseline."""
import bench


def _profile(root, name, hash_, traffic):
    d = root / "profiles"
    d.mkdir(exist_ok=True)
    (d / f"{name}.md").write_text(f"# x\n\nkernel_source_hash: {hash_} (note)\n"
                                  f"traffic_bytes_per_launch: {traffic}\n")


def test_recorded_traffic_only_for_the_captured_source(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    src = tmp_path / "k.cu"
    src.write_text("__global__ void f() { int a = 1; }  // first form\n")
    h = bench.kernel_source_hash(["k.cu"])
    _profile(tmp_path, "p", h, 123456789)
    assert bench.recorded_traffic("p", ["k.cu"]) == 123456789.0
    # a comment-only or whitespace edit keeps the figure ...
    src.write_text("/* doc */\n__global__ void f() {\n  int a = 1;\n}  // reworded\n")
    assert bench.kernel_source_hash(["k.cu"]) == h
    assert bench.recorded_traffic("p", ["k.cu"]) == 123456789.0
    # ... a code change retires it
    src.write_text("__global__ void f() { int a = 2; }\n")
    assert bench.recorded_traffic("p", ["k.cu"]) is None
    assert bench.recorded_traffic("missing", ["k.cu"]) is None


def test_host_cpu_names_the_processor():
    name = bench.host_cpu()
    assert isinstance(name, str) and name.strip() and name != "unknown"
