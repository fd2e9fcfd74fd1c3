"""Host logic of bench.py that decides what its JSON line reports (no GPU).

- The DRAM traffic of a kernel comes from the committed ncu table only when
  the table's line was taken on the kernel's current source (its SHA-256
  prefix), and is scaled to the bench's launch by the ratio of algorithmic
  bytes; the statistics step picks the table line of the kernel that runs
  (two CTAs per SM up to 128 candidate blocks per row, one CTA beyond).
- A kernel timed inside the long step is held to the sustained bf16 peak, a
  kernel timed alone to the burst peak; both fractions are reported, and the
  HBM kernels are held to the measured copy bandwidth.
- The peaks come from MEASURED_PEAKS.json when present, else the fallback.
"""
import hashlib
import json
import os
import sys
import types

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
import bench  # noqa: E402

SOURCES = {"stats2": "mf_stats2_tc.cu", "stats": "mf_stats_tc.cu", "pack": "mf_pack_tc.cu",
           "retrieve": "mf_retrieve_team.cu"}


@pytest.fixture
def fake_root(tmp_path, monkeypatch):
    csrc = tmp_path / "cross_model_attention_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    for name, f in SOURCES.items():
        (csrc / f).write_text(f"// source of {name}\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    return tmp_path


def sha(root, name):
    path = os.path.join(root, "cross_model_attention_gb300", "csrc", SOURCES[name])
    return hashlib.sha256(open(path, "rb").read()).hexdigest()[:16]


def write_table(root, lines):
    (root / "profiles" / "ncu_traffic.txt").write_text(
        "# kernel sha dram alg\n" + "\n".join(lines) + "\n")


def test_traffic_needs_a_line_on_the_current_source(fake_root):
    assert bench.traffic_for("retrieve", 1e9) is None  # no table
    write_table(fake_root, [f"retrieve {'0' * 16} 700 650"])
    assert bench.traffic_for("retrieve", 1e9) is None  # stale source
    write_table(fake_root, [f"retrieve {sha(fake_root, 'retrieve')} 700 650"])
    assert bench.traffic_for("retrieve", 650.0) == pytest.approx(700.0)
    # scaled by the ratio of algorithmic bytes
    assert bench.traffic_for("retrieve", 1300.0) == pytest.approx(1400.0)
    (fake_root / "cross_model_attention_gb300" / "csrc" / SOURCES["retrieve"]).write_text("// changed\n")
    assert bench.traffic_for("retrieve", 650.0) is None


def test_statistics_traffic_follows_the_kernel_that_runs(fake_root):
    write_table(fake_root, [f"stats {sha(fake_root, 'stats2')} 110 100",
                            f"stats {sha(fake_root, 'stats')} 150 100"])
    assert bench.traffic_for("stats", 100.0, max_blocks=128) == pytest.approx(110.0)
    assert bench.traffic_for("stats", 100.0, max_blocks=129) == pytest.approx(150.0)


def test_the_committed_table_parses():
    # every line of the committed table names a kernel, a 16-hex-digit
    # source hash and two positive byte counts
    path = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    n = 0
    for line in open(path):
        if line.startswith("#") or not line.strip():
            continue
        kernel, digest, dram, alg = line.split()[:4]
        assert kernel in ("stats", "pack", "retrieve")
        assert len(digest) == 16 and int(digest, 16) >= 0
        assert float(dram) > 0 and float(alg) > 0
        n += 1
    assert n >= 3


def roofs(long_step):
    w = types.SimpleNamespace(B=64, seqlens=[4096], T=4096, sender_heads=40, sender_kv_heads=40, d=128)
    prof = {"stats": (10, 1.0), "pack": (10, 2.0), "retrieve": (20, 4.0)}  # (launches, total ms)
    peaks = {"hbm_gbs": 6000.0, "bf16_tflops": 2000.0, "bf16_tflops_sustained": 1600.0}
    # 10 layers: 1 TFLOP of Q.K^T per layer; 0.1 ms per statistics launch
    return bench.rooflines_of(w, prof, 10, 2.0e9 * 20, 1.0e12 * 10, 1.5e9 * 10, peaks,
                              "of measured", long_step)


def test_in_step_kernels_are_held_to_the_sustained_peak(fake_root):
    r = roofs(long_step=True)
    st = r["stats"]
    assert st["achieved"] == pytest.approx(1.0e12 / 1.0e-4 / 1e12)  # 10,000 TFLOP/s
    assert st["peak"] == 1600.0 and "sustained" in st["peak_source"]
    assert st["frac"] == pytest.approx(st["achieved"] / 1600.0)
    assert st["frac_of_burst"] == pytest.approx(st["achieved"] / 2000.0)
    alone = roofs(long_step=False)["stats"]
    assert alone["peak"] == 2000.0 and alone["frac"] == pytest.approx(alone["frac_of_burst"])


def test_hbm_kernels_use_the_measured_copy_bandwidth(fake_root):
    r = roofs(long_step=True)
    ret = r["retrieve"]
    # 2 GB per launch in 0.2 ms
    assert ret["algorithmic_bytes_per_launch"] == pytest.approx(2.0e9)
    assert ret["achieved"] == pytest.approx(2.0e9 / 2.0e-4 / 1e9)
    assert ret["frac"] == pytest.approx(ret["achieved"] / 6000.0)
    assert ret["frac_of_8TBs_nominal"] == pytest.approx(ret["achieved"] / 8000.0)
    assert ret["traffic"] is None  # no table in the fake root
    pk = r["pack"]
    assert pk["achieved"] == pytest.approx(1.5e9 / 2.0e-4 / 1e9)


def test_peaks_come_from_the_measured_file_else_the_fallback(fake_root):
    peaks, src = bench.load_peaks()
    assert src == "fallback" and peaks == bench.FALLBACK_PEAKS
    (fake_root / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 1.0, "bf16_tflops": 2.0}))
    peaks, src = bench.load_peaks()
    assert src == "measured" and peaks["hbm_gbs"] == 1.0
