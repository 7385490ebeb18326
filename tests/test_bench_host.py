"""Host logic of bench.py (no GPU): the algorithmic byte count, the weak-
scaling value, and the rule that the profiled DRAM traffic is reported only
while the kernel sources are those it was captured on."""
import bench


def test_algorithmic_bytes_match_the_definition():
    # (N + 3) reads + 2 writes of M*H BF16 values, plus w and gamma
    M, N, H = 8192, 12, 7168
    assert bench.algorithmic_bytes(M, N, H) == (N + 5) * M * H * 2 + 4 * H == 1_996_517_376
    assert bench.algorithmic_bytes(M, N, H, has_add2=False) == (N + 4) * M * H * 2 + 4 * H


def test_weak_scaling_value_counts_every_rank():
    nb = bench.algorithmic_bytes(8192, 12, 7168)
    one = bench.weak_scaling_value(nb, 1, 10, 1.0)
    assert abs(bench.weak_scaling_value(nb, 4, 10, 1.0) - 4 * one) < 1e-9 * one


def test_profiled_traffic_follows_the_kernel_sources(tmp_path, monkeypatch):
    digest = bench.kernel_source_digest()
    f = tmp_path / "traffic.txt"
    f.write_text(f"# summary\nkernel_source_digest = {digest}\ndram_bytes_per_launch = 1234\n")
    monkeypatch.setattr(bench, "PROFILE_TRAFFIC", str(f))
    assert bench.profiled_traffic() == 1234
    f.write_text("kernel_source_digest = 0000000000000000\ndram_bytes_per_launch = 1234\n")
    assert bench.profiled_traffic() is None
    monkeypatch.setattr(bench, "PROFILE_TRAFFIC", str(tmp_path / "missing.txt"))
    assert bench.profiled_traffic() is None

