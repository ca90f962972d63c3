"""Host logic of bench.py that needs no GPU: the algorithmic work each
workload's throughput and roofline divide by, the per-step percentiles, the
whole-job value, and the rule that a DRAM traffic figure is reported only
while the kernel sources it was captured on are unchanged."""
import json
import os

import pytest

import bench


@pytest.mark.parametrize("name,work", [
    # 2 M N K for the Linear chains (x[M,1024] W[4096,1024]; x[1024,8192] W[8192,8192])
    ("linear_gn_m32768", 2 * 32768 * 4096 * 1024),      # 274.878 GFLOP
    ("linear_gn_m256", 2 * 256 * 4096 * 1024),          # 2.147 GFLOP
    ("linear_lse_m1024", 2 * 1024 * 8192 * 8192),       # 137.439 GFLOP
    # 2 B L C C k for the dilated Conv1d (x[32,256,4096], k 3)
    ("ln_dconv1d_b32", 2 * 32 * 4096 * 256 * 256 * 3),  # 51.540 GFLOP
    # ConvTranspose3d: x read once + out [128,16,31,63,63] written once, fp32
    ("convt3d_n128", 4 * (128 * 3 * 16 * 32 * 32 + 128 * 16 * 31 * 63 * 63)),  # 1033.1 MB
])
def test_algorithmic_work_per_step(name, work):
    wl = bench.make_workload(name)
    assert wl.work_per_step() == work
    assert wl.kernel_work() == work
    assert wl.scale() == (1e9 if wl.unit == "GB/s" else 1e12)
    assert wl.bound == ("hbm" if name == "convt3d_n128" else "tensor")


def test_convt3d_output_shape_is_the_pages():
    assert bench.make_workload("convt3d_n128").out_shape == (128, 16, 31, 63, 63)


def test_step_percentiles():
    got = bench.step_percentiles([float(v) for v in (7, 3, 9, 1, 5, 2, 8, 4, 10, 6)])
    assert got == {"median": 5.5, "p10": 1.0, "p90": 9.0, "n": 10}
    assert bench.step_percentiles([2.5]) == {"median": 2.5, "p10": 2.5, "p90": 2.5, "n": 1}
    assert bench.step_percentiles([]) is None


def test_job_value_counts_every_rank():
    # 275 GFLOP per rank, 4 ranks, 1 ms for the slowest: 1100 TFLOP/s for the job
    assert bench.job_value(275e9, 4, 1.0, 1e12) == pytest.approx(1100.0)


def test_traffic_only_on_the_sources_it_was_captured_on(tmp_path, monkeypatch):
    csrc = tmp_path / "conv_activation_normalization_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "k.cu").write_text("kernel v1\n")
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))

    class W:
        name = "w"
        sources = ("k.cu",)

    assert bench._kernel_traffic(W()) is None  # no summary committed
    sha = bench.kernel_source_sha(W.sources)
    (tmp_path / "profiles" / "traffic.json").write_text(
        json.dumps({"w": {"traffic_bytes_per_launch": 123, "source_sha": sha}}))
    assert bench._kernel_traffic(W()) == 123
    (csrc / "k.cu").write_text("kernel v2\n")  # the kernel changed since the capture
    assert bench._kernel_traffic(W()) is None


def test_committed_traffic_entries_name_known_workloads():
    p = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "profiles", "traffic.json")
    d = json.load(open(p))
    assert set(d) <= set(bench.ALL)
    for name, e in d.items():
        # traffic = dram__bytes_read.sum + dram__bytes_write.sum of one launch, within a
        # factor of two of the launch's algorithmic bytes (a capture of another kernel or
        # of a cut-down case would fall outside; the output lines still in L2 when the
        # kernel ends are never written back inside the launch, so it can be below)
        assert e["traffic_bytes_per_launch"] == e["dram_read_bytes"] + e["dram_write_bytes"]
        assert len(e["source_sha"]) == 16
        algo = algo_bytes(name, bench.make_workload(name).kernel_work())
        assert 0.5 * algo < e["traffic_bytes_per_launch"] < 2.0 * algo, (name, e["traffic_bytes_per_launch"], algo)


def algo_bytes(name, work):
    """Algorithmic DRAM bytes of one launch of each workload's dominant kernel."""
    M, K, N = {"linear_gn_m32768": (32768, 1024, 4096), "linear_gn_m256": (256, 1024, 4096),
               "linear_lse_m1024": (1024, 8192, 8192)}.get(name, (0, 0, 0))
    if name == "linear_gn_m256":  # x, W, out: at 64-column tiles the GEMM computes both lo planes itself
        return 4 * (M * K + N * K + M * N)
    if name.startswith("linear_gn"):  # x and its lo plane, W and its lo plane, out
        return 4 * (2 * M * K + 2 * N * K + M * N)
    if name == "linear_lse_m1024":  # x and its lo plane, W (the GEMM computes W's lo plane; the partials are small)
        return 4 * (2 * M * K + N * K)
    if name == "ln_dconv1d_b32":  # the activations' raw plane (the GEMM computes lo), W planes, x (residual), out
        B, C, L = 32, 256, 4096
        return 4 * (B * C * L + 2 * C * C * 3 + 2 * B * C * L)
    return work  # convt3d: x once + out once


def test_host_threads_follow_the_blas_pool_or_the_environment(monkeypatch):
    import sys
    n = len(os.sched_getaffinity(0))
    assert 1 <= bench.host_threads() <= n
    # without threadpoolctl (as on hosts that lack it) the variables decide, in OpenBLAS's order
    monkeypatch.setitem(sys.modules, "threadpoolctl", None)
    for v in ("OPENBLAS_NUM_THREADS", "GOTO_NUM_THREADS", "OMP_NUM_THREADS"):
        monkeypatch.delenv(v, raising=False)
    assert bench.host_threads() == n
    monkeypatch.setenv("OMP_NUM_THREADS", "1")  # what torchrun sets
    assert bench.host_threads() == 1
    monkeypatch.setenv("OPENBLAS_NUM_THREADS", "2")
    assert bench.host_threads() == min(n, 2)
    monkeypatch.setenv("OPENBLAS_NUM_THREADS", "100000")
    assert bench.host_threads() == n


def test_launches_per_step_match_the_committed_launch_lists():
    # the bench's per-step launch count (its gpu_launches claim) against the
    # ncu launch lists under profiles/ (3xTF32 mode): the library's launches
    # over the dominant kernel's, which runs once per step
    import json
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    traffic = json.load(open(os.path.join(root, "profiles", "traffic.json")))
    for name, entry in traffic.items():
        counts = {}
        for line in open(os.path.join(root, "profiles", f"{name}_launches.md")):
            cells = [c.strip() for c in line.split("|")]
            if len(cells) > 3 and cells[1].startswith("`") and not cells[1].startswith("`at::"):
                counts[cells[1].strip("`")] = int(cells[2])
        assert entry["kernel"] in counts, (name, entry["kernel"])
        assert sum(counts.values()) % counts[entry["kernel"]] == 0, (name, counts)
        assert sum(counts.values()) // counts[entry["kernel"]] == bench.launches_per_step(name, "3xtf32"), \
            (name, counts)
