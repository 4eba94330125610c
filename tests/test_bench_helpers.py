"""bench.py's measurement arithmetic, on the CPU: the roofline figures it derives from per-kernel
times, the expert sizes of a narrowed FFN, and the DRAM traffic it reads from the committed
ncu summaries (only while the summarised kernel's source is unchanged)."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


@pytest.fixture(autouse=True)
def _k3_width():
    yield
    bench._set_ffn_width(1536)


def test_expert_sizes_follow_the_packed_byte_rule():
    # 17/32 bytes per weight (a nibble plus a 1/32 share of a scale byte): the K3 expert count
    assert (bench.EXPERT_BYTES, bench.GATEUP_BYTES, bench.DOWN_BYTES) == (17_547_264, 11_698_176, 5_849_088)
    bench._set_ffn_width(128)
    assert bench.F == 128 and bench.EXPERT_BYTES == 3 * 128 * 7168 * 17 // 32
    assert bench.GATEUP_BYTES == 2 * bench.DOWN_BYTES
    with pytest.raises(SystemExit):
        bench._set_ffn_width(100)


def test_decode_roofline_is_expert_bytes_over_gateup_time():
    # 16 experts' gate/up bytes in 43.5 us, 5 launches timed
    prof = {"gemm_gu": (0.0, 0), "gemm_dn": (0.0, 0), "gateup": (5 * 0.0435, 5), "down": (5 * 0.028, 5),
            "combine": (5 * 0.0062, 5)}
    r = bench._roofline(prof, 1, 16, 6494.9, 1801.9, "measured")
    expect = 16 * 11_698_176 / 43.5e-6 / 1e9
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert r["achieved"] == pytest.approx(expect, abs=0.1)
    assert r["frac"] == pytest.approx(expect / 6494.9, abs=1e-4)
    assert r["algorithmic_bytes_per_launch"] == 16 * 11_698_176
    assert r["down_kernel_gbs"] == pytest.approx(16 * 5_849_088 / 28e-6 / 1e9, abs=0.1)
    assert r["combine_kernel_gbs"] == pytest.approx((16 * 7168 * 4 + 7168 * 4) / 6.2e-6 / 1e9, abs=0.1)


def test_prefill_roofline_is_gateup_flops_over_gemm_time():
    prof = {"gemm_gu": (2.85, 1), "gemm_dn": (1.74, 1), "gateup": (0.0, 0), "down": (0.0, 0),
            "combine": (0.31, 1)}
    r = bench._roofline(prof, 4096, 32, 6494.9, 1801.9, "measured")
    flops = 4.0 * 1536 * 7168 * 4096 * 16  # gate and up: 2 * 2 * f * d per pick
    assert r["bound"] == "tensor" and r["algorithmic_flops_per_launch"] == flops
    assert r["achieved"] == pytest.approx(flops / 2.85e-3 / 1e12, abs=0.1)
    assert r["frac"] == pytest.approx(flops / 2.85e-3 / 1e12 / 1801.9, abs=1e-4)
    assert r["down_gemm_tflops"] == pytest.approx(flops / 2 / 1.74e-3 / 1e12, abs=0.1)
    # the combine reads every pick's fp32 row and writes y: 2.0 GB at the copy peak
    assert r["combine_kernel_gbs"] == pytest.approx((4096 * 16 + 4096) * 7168 * 4 / 0.31e-3 / 1e9, abs=0.1)


def test_traffic_is_read_only_while_the_kernel_source_matches(tmp_path, monkeypatch):
    src = tmp_path / "kernel.cu"
    src.write_text("// kernel\n")
    (tmp_path / "profiles").mkdir()
    summary = tmp_path / "profiles" / "k.txt"
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    summary.write_text(f"# header\nsource_sha256_16: {bench._source_hash('kernel.cu')}\n"
                       "dram_bytes_per_launch: 187563520\n")
    assert bench._traffic_from_profile("kernel.cu", "k.txt") == 187563520
    src.write_text("// kernel, changed\n")
    assert bench._traffic_from_profile("kernel.cu", "k.txt") is None
    assert bench._traffic_from_profile("kernel.cu", "missing.txt") is None


def test_committed_decode_profiles_parse():
    # the committed summaries carry the fields bench.py reads
    for name in ("gateup_decode_k3_t1.txt", "gateup_decode_k3_t64.txt", "gemm_gu_prefill_k3_t4096.txt"):
        kv = {}
        with open(os.path.join(ROOT, "profiles", name)) as fh:
            for ln in fh:
                if ":" in ln and not ln.startswith("#"):
                    a, b = ln.split(":", 1)
                    kv[a.strip()] = b.strip()
        assert len(kv["source_sha256_16"]) == 16
        assert int(kv["dram_bytes_per_launch"]) > 0
