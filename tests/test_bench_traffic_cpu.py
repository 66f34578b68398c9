"""The DRAM-traffic figures bench.py reports: tied to the kernel sources they were captured from."""
import os
import sys

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402


def test_stored_traffic_matches_current_sources():
    """Every stored capture was taken on the kernel sources in this tree, so the bench line reports it."""
    for (workload, kernel), (h, nbytes) in bench.KERNEL_TRAFFIC.items():
        assert h == bench.csrc_hash(bench.KERNEL_SOURCES[kernel]), (workload, kernel)
        assert bench.kernel_traffic(workload, kernel) == nbytes


def test_changed_sources_report_no_traffic(monkeypatch):
    """A kernel edited since its capture reports null traffic instead of a stale figure."""
    monkeypatch.setattr(bench, "csrc_hash", lambda files=None: "0" * 16)
    for workload, kernel in bench.KERNEL_TRAFFIC:
        assert bench.kernel_traffic(workload, kernel) is None
    assert bench.kernel_traffic("no_such_workload", "attn") is None


def test_hash_ignores_comments(tmp_path, monkeypatch):
    """Comments and blank space do not change the hash; code does."""
    d = tmp_path / "block_quantized_token_gb300" / "csrc"
    d.mkdir(parents=True)
    (tmp_path / "include").mkdir()
    (tmp_path / "include" / "er.h").write_text("int f(void);\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    (d / "k.cu").write_text("int a = 1; // one\n/* block\n comment */ int b = 2;\n")
    h0 = bench.csrc_hash(("k.cu",))
    (d / "k.cu").write_text("int a = 1;   // changed comment\n\n int b = 2;\n")
    assert bench.csrc_hash(("k.cu",)) == h0
    (d / "k.cu").write_text("int a = 1; int b = 3;\n")
    assert bench.csrc_hash(("k.cu",)) != h0
