"""Host-side logic of the benchmark that needs no GPU: workload selection, the
80 GB admissibility figure of the sweep, byte accounting and the oracle
sample shapes."""
import sys
import os

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from paged_fp8_kv_decode_gb300 import workloads as W  # noqa: E402


def test_sweep_admissible_batch_for_an_80_gb_pool_over_32_layers():
    # 32,768 tokens x 32 layers x (2 x 8 heads x 128 dims x 2 B) = 4.29 GB per
    # BF16 sequence -> 18 fit in 80 GB; FP8 (+ two fp32 scales per 16-token
    # unit and kv head) = 2.15 GB -> 37 fit.
    assert bench.sweep_admissible(W.spec_sweep(1, "bf16")) == 18
    assert bench.sweep_admissible(W.spec_sweep(1, "fp8")) == 37


def test_workload_spec_names_and_sizes():
    a = bench.parse_args(["--workload", "sweep", "--batch", "16", "--kv-dtype", "bf16"])
    s = bench.workload_spec(a)
    assert (s.B, s.kv_dtype, int(s.lens[0])) == (16, "bf16", 32768)
    assert s.num_pages == W.sweep_pool_pages("bf16")
    s = bench.workload_spec(bench.parse_args(["--workload", "long"]))
    assert s.split_tokens == 4096 and list(s.lens) == [131072, 262144, 393216, 524288]
    s = bench.workload_spec(bench.parse_args(["--workload", "evict"]))
    assert s.per_head and s.lens.shape == (16, 8) and s.stale_per_mille == 1.0
    s = bench.workload_spec(bench.parse_args([]))
    assert s.name == "llama8b" and s.B == 32 and s.append
    s = bench.workload_spec(bench.parse_args(["--workload", "sweep", "--head-dim", "64"]))
    assert s.D == 64 and s.Hq == 32 and int(s.lens[0]) == 32768
    # an admissible batch counts the head dim: half the bytes per token at 64
    assert bench.sweep_admissible(s) == 74


def test_sample_shape_bounds_the_oracle_work():
    for spec in (W.spec_llama8b("full"), W.spec_long("full"), W.spec_evict("full"),
                 W.spec_sweep(64, "fp8")):
        n, nh = bench._sample_shape(spec)
        assert 1 <= n <= min(4, spec.B) and 1 <= nh <= spec.Hkv
        lens = np.asarray(spec.lens).astype(np.int64)
        per_req = lens if lens.ndim == 1 else lens.max(axis=1)
        assert int(per_req[:n].sum()) * nh <= 600_000 or (n == 1 and nh == 1)


def test_aborted_requests_drop_their_kv_and_scales_but_not_their_tags():
    class FakeDB:
        pass
    from paged_fp8_kv_decode_gb300.device_batch import DeviceBatch
    spec = W.spec_evict("small")
    db = FakeDB()
    db.spec, db.batch = spec, W.make_batch(spec)
    db.cache = type("C", (), {"page_tags": object()})()
    for name in ("_lens", "kv_bytes", "algorithmic_bytes"):
        setattr(db, name, getattr(DeviceBatch, name).__get__(db))
    lens = db.batch.lens_bh("seq").astype(np.int64)
    pages = (lens + 15) // 16
    skip = np.zeros(spec.B, bool)
    skip[1] = True
    full = db.algorithmic_bytes()
    part = db.algorithmic_bytes(skip=skip)
    kv1 = int(lens[1].sum()) * spec.D * 2
    assert full - part == kv1 + 8 * int(pages[1].sum())
    assert db.algorithmic_bytes(tags=False) == full - 8 * int(pages.sum())


def test_clock_summary_reads_load_samples_and_throttle_reasons(tmp_path):
    """nvidia-smi rows (index, sm MHz, max MHz, power W, active mask, hw_slowdown,
    hw_thermal, sw_thermal, sw_power_cap): the median SM clock is taken over
    the samples under load (above 200 W), reasons over the same samples."""
    p = tmp_path / "clocks.csv"
    p.write_text("\n".join([
        "0, 2070, 2070, 90.0, 0x0, Not Active, Not Active, Not Active, Not Active",   # idle
        "0, 2070, 2070, 650.5, 0x0, Not Active, Not Active, Not Active, Not Active",
        "0, 1995, 2070, 1390.0, 0x4, Not Active, Not Active, Not Active, Active",
        "0, 2055, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "garbage line",
    ]) + "\n")
    s = bench.ClockSampler(0, str(p)).summary()
    assert s["samples"] == 3 and s["sm_mhz"] == 2055.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"] and s["power_w_max"] == 1390.0


def test_clocks_path_defaults_to_a_temporary_file(tmp_path):
    a = bench.parse_args([])
    path = bench.clocks_path(a)
    assert os.path.exists(path) and "pfkv_clocks_" in os.path.basename(path)
    os.remove(path)
    a = bench.parse_args(["--clocks-csv", str(tmp_path / "sub" / "c.csv")])
    assert bench.clocks_path(a) == str(tmp_path / "sub" / "c.csv")
    assert os.path.isdir(tmp_path / "sub")


def test_roofline_traffic_comes_from_the_capture_of_the_same_source(tmp_path, monkeypatch):
    """roofline.traffic is the committed capture's DRAM bytes scaled to the
    run's algorithmic bytes, and null once the kernel source has changed, or
    for a workload with no capture of its own."""
    for name in ("decode_split_pers_llama8b_fp8.md", "decode_split_pers_long_fp8.md"):
        assert os.path.exists(os.path.join(ROOT, "profiles", name)), name
    src = tmp_path / "k.cu"
    src.write_text("kernel v1\n")
    import hashlib
    digest = hashlib.sha256(b"kernel v1\n").hexdigest()[:16]
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "s.md").write_text(
        "text: ignored\n    kernel_source: k.cu\n"
        f"    kernel_source_sha256_16: {digest}\n"
        "    dram_bytes_per_launch: 1020\n    algorithmic_bytes_per_launch: 1000\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profiled_traffic(2000, "s.md") == pytest.approx(2040)
    assert bench.profiled_traffic(2000, "missing.md") is None
    monkeypatch.setattr(bench, "WORKLOAD_PROFILES", {"long": "s.md"})
    assert bench.workload_traffic("long", 500) == 510
    assert bench.workload_traffic("sweep", 500) is None
    src.write_text("kernel v2\n")
    assert bench.profiled_traffic(2000, "s.md") is None
    assert bench.workload_traffic("long", 500) is None


def test_dtype_label_follows_the_kernel_path():
    llama = W.spec_llama8b("small")
    assert bench.path_dtype(llama) == bench.FP8_DTYPE
    assert bench.path_dtype(W.spec_tiny()) == bench.BF16_MMA_DTYPE  # head_dim 64: tensor cores too
    assert bench.path_dtype(W.spec_sweep(8, "bf16", "small")) == bench.BF16_MMA_DTYPE
