"""Host logic of bench.py that its reported figures rest on, without a GPU:
the algorithmic bytes of each segment (the roofline numerators) restated as
closed forms of the workload shapes, the roofline arithmetic, and the rule
that a captured DRAM traffic figure is reported only while the kernel's
sources are the captured ones."""
import os
import shutil

import pytest

import bench
import workloads


def test_headline_algorithmic_bytes():
    """CSA decode, B = 32 at 128K: 32768 complete blocks a sequence; the
    indexer streams bf16 keys (128 dims) plus 64 query heads and weights;
    the attention reads 1024 selected + 128 window rows of 1 KiB plus q and
    out (64 heads x 512 bf16 each); the top-k reads the float32 score rows."""
    w = workloads.CSA_DECODE_128K
    seg, step = bench.algorithmic(w, 1024)
    n = 131072 // 4
    assert seg["indexer"]["bytes"] == 32 * (n * 128 * 2 + 64 * 128 * 2 + 64 * 4) == 268967936
    assert seg["attention"]["bytes"] == 32 * ((1024 + 128) * 1024 + 2 * 64 * 512 * 2) == 41943040
    assert seg["topk"]["bytes"] == 32 * n * 4
    assert step > seg["indexer"]["bytes"] + seg["attention"]["bytes"]  # plus the append


def test_hca_and_low_bit_key_bytes():
    w = workloads.HCA_DECODE_1M
    seg, _ = bench.algorithmic(w, 1024)
    n = 1048576 // 128
    assert seg["attention"]["bytes"] == 32 * ((n + 128) * 1024 + 2 * 64 * 512 * 2) == 276824064
    # E4M3 keys: 128 code bytes and a float32 scale; FP4: 64 code bytes and 4 exponent bytes
    for fmt, per_key in (("fp8", 132), ("fp4", 68)):
        wq = workloads.CSA_DECODE_128K.replace(idx_fmt=fmt)
        seg, _ = bench.algorithmic(wq, 1024)
        assert seg["indexer"]["bytes"] == 32 * (32768 * per_key + 64 * 128 * 2 + 64 * 4)


def test_roofline_arithmetic():
    peaks = {"hbm_gbs": 6500.0, "bf16_tflops": 1700.0, "sm_max_mhz": 2032.0, "source": "measured"}
    r = bench._roofline("indexer", {"bound": "hbm", "bytes": 65_000_000}, 0.01, peaks, None)
    assert r["achieved"] == pytest.approx(6500.0) and r["frac"] == pytest.approx(1.0)
    r = bench._roofline("attention", {"bound": "tensor", "flops": 17_000_000_000}, 0.01, peaks, 123)
    assert r["unit"] == "TFLOP/s" and r["frac"] == pytest.approx(1.0) and r["traffic"] == 123


def test_captured_traffic_follows_the_sources(tmp_path, monkeypatch):
    key = ("csa_decode_bf16_b32_128k", "indexer")
    files, _, nbytes = bench.CAPTURED_TRAFFIC[key]
    if bench.captured_traffic(*key) is None:
        pytest.skip("the indexer's sources changed since its capture")
    assert bench.captured_traffic(*key) == nbytes
    # the same files with one byte more: no figure
    src = os.path.join(bench.ROOT, "long_context_compressed_17_b300", "csrc")
    dst = tmp_path / "long_context_compressed_17_b300" / "csrc"
    dst.mkdir(parents=True)
    for f in files:
        shutil.copy(os.path.join(src, f), dst / f)
    with open(dst / files[0], "ab") as fh:
        fh.write(b"\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.captured_traffic(*key) is None
    assert bench.captured_traffic("no_such_workload", "indexer") is None
