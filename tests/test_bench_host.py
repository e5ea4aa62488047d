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


def test_clock_normalised_fraction():
    peaks = {"clocks_under_load": {"sm_mhz_median": 1500.0}}
    # a run at a higher clock than the peak's is held to the peak scaled up
    assert abs(bench.clock_normalised(1800.0, 1800.0, {"sm_mhz": 1800.0}, peaks) - 1500.0 / 1800.0) < 1e-12
    assert bench.clock_normalised(1.0, 1.0, None, peaks) is None
    assert bench.clock_normalised(1.0, 1.0, {"sm_mhz": 1800.0}, {}) is None


def test_cpu_baseline_names_threads(tmp_path):
    """Both oracle timings run (in child processes) and say how many threads
    they used; the headline value is the single-threaded one."""
    from indexer_topk_long_gb300 import datagen
    inp = datagen.make_indexer_inputs(T=6, first_pos=300, S=306, H=4, d=16, seed=2)
    rec = bench.cpu_baseline_record(inp, 16, 2, 3)
    assert rec["cores"] == 1 and rec["single_thread"]["threads"] == 1
    assert rec["value"] == rec["single_thread"]["value"] > 0
    assert rec["all_cores"]["threads"] >= 1 and rec["all_cores"]["value"] > 0
    assert bench._sample_queries(6, 3) == [0, 2, 5]
