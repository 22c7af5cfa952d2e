"""Host-side logic of bench.py that needs no GPU: the recorded DRAM traffic is
reported only while the kernel sources it was captured with are unchanged, and
the oracle's CPU sample is sized to its time budget and counts its own work."""
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
    # a fake oracle leg whose sized sample takes 0.5 s a pass
    calls = []

    class FakeLeg:
        def __init__(self, config):
            calls.append(("config", config))

        def size_for(self, budget_s):
            calls.append(("size_for", budget_s))
            return 0.25

        def prepare(self, f):
            calls.append(("prepare", f))

        def run(self):
            calls.append("run")
            return 0.5

        def value(self, seconds):
            return 2.0 / seconds

        def describe(self):
            return "sample"

        def cores(self):
            return 4

    clock = iter(range(1000))
    monkeypatch.setattr(bench, "OracleLeg", FakeLeg)
    monkeypatch.setattr(bench.time, "time", lambda: float(next(clock)))
    value, secs, sample, cores = bench.oracle_sample("q4_1", 10.0)
    # half the budget sizes the sample, one pass measures it, then whole
    # passes fill the other half: 5 s / 0.5 s = 10 passes
    assert calls[:4] == [("config", "q4_1"), ("size_for", 5.0), ("prepare", 0.25), "run"]
    assert calls[4:] == ["run"] * 10
    assert sample.startswith("10 pass(es) of the sample")
    assert cores == 4 and secs > 0 and value > 0


def test_oracle_leg_counts_the_work_of_its_sample():
    # the MLP pair at a 1/64 sample: every shard of W1 keeps ceil(2752/64) = 43
    # rows, W2 keeps ceil(4096/64) = 64 rows, all 512 token rows
    leg = bench.OracleLeg("mlp")
    leg.prepare(1.0 / 64)
    T, D, F, N = 512, 4096, 11008, 4
    assert leg.work == 2.0 * T * D * 43 * N + 2.0 * T * F * 64
    assert leg.full == 2.0 * 2 * T * D * F
    assert leg.unit() == "TFLOP/s"
    assert leg.cores() >= 1
    assert leg.run() > 0
    assert leg.value(1.0) == leg.work / 1e12


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
