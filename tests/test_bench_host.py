"""Host-side logic of bench.py that needs no GPU: the recorded DRAM traffic is
reported only while the kernel sources it was captured with are unchanged, and
the oracle's CPU sample is sized to its time budget."""
import bench


def test_traffic_reported_only_for_matching_sources(monkeypatch):
    key = ("mlp", "tp_sharded_to_all")
    assert key in bench.TRAFFIC
    fam = bench.config_family("mlp")
    assert fam == "umma"
    monkeypatch.setitem(bench.TRAFFIC_SOURCES, fam, bench.kernel_sources_hash(fam))
    assert bench.traffic_for(*key) == bench.TRAFFIC[key]
    monkeypatch.setitem(bench.TRAFFIC_SOURCES, fam, "0" * 16)
    assert bench.traffic_for(*key) is None


def test_every_traffic_entry_names_a_known_family():
    for (config, _call), nbytes in bench.TRAFFIC.items():
        assert bench.config_family(config) in bench.TRAFFIC_SOURCES
        assert nbytes > 0


def test_family_hash_covers_the_shared_split_sum():
    # the ordered split sum serves the 4-bit and mxfp8 kernels: a change to it
    # must invalidate their recorded traffic
    assert "k_split.cu" in bench.COMMON_SOURCES


def test_oracle_sample_fills_its_budget_with_whole_passes(monkeypatch):
    # a fake oracle run: 1 ms per row plus 50 ms per call
    calls = []

    class FakeMLP:
        total_rows, per_row, desc = 512, 1.0, "rows"

        def __init__(self):
            import types
            self.oracle = types.SimpleNamespace(num_threads=lambda: 4)

        def run(self, rows):
            calls.append(rows)
            return 0.05 + 0.001 * rows

        seconds_per_row = bench.OracleMLP.seconds_per_row
        rows_for = bench.OracleMLP.rows_for

    clock = iter(range(1000))
    monkeypatch.setattr(bench, "OracleMLP", FakeMLP)
    monkeypatch.setattr(bench.time, "time", lambda: float(next(clock)))
    value, secs, sample, cores = bench.oracle_sample(10.0)
    # calibration: one 64-row pass (1.78 ms a row); 10 s covers the whole batch
    # (512 rows, 0.91 s a pass by that estimate), so 10 whole passes follow
    assert calls[0] == 64
    assert calls[1:] == [512] * 10
    assert sample.startswith("10 pass(es) of 512 of 512")
    assert cores == 4 and secs > 0 and value > 0


def test_source_hash_ignores_comments_but_not_code(tmp_path, monkeypatch):
    import shutil
    src = bench.os.path.join(bench.ROOT, "sharded_gemm_gb300", "csrc")
    dst = tmp_path / "sharded_gemm_gb300" / "csrc"
    shutil.copytree(src, dst)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench.kernel_sources_hash("umma")
    f = dst / "k_umma.cu"
    text = f.read_text()
    f.write_text(text + "\n// a note\n/* and a\n   block note */\n")
    assert bench.kernel_sources_hash("umma") == h0
    f.write_text(text + "\nstatic int unused_probe_value;\n")
    assert bench.kernel_sources_hash("umma") != h0
    # the shared split sum belongs to every family
    f.write_text(text)
    g = dst / "k_split.cu"
    g.write_text(g.read_text() + "\nstatic int unused_probe_value;\n")
    assert bench.kernel_sources_hash("umma") != h0
