"""Host-side arithmetic of bench.py on CPU: the roofline fields of a launch, the use of the
committed ncu traffic figures (only for the kernel sources they were taken on), and the
algorithmic bytes of the decode batch."""

import json
import sys
from pathlib import Path

import pytest
import torch

ROOT = Path(__file__).resolve().parent.parent
sys.path.insert(0, str(ROOT))

import bench  # noqa: E402
from workloads import gathered_bytes  # noqa: E402

PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def test_roofline_fields_below_64_heads_are_hbm_bound():
    r = bench.roofline_fields(8, 75_497_472.0, 1152, 0.020, PEAKS)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert r["achieved"] == pytest.approx(75_497_472.0 / 20e-6 / 1e9)
    assert r["frac"] == pytest.approx(r["achieved"] / 6800.0)


def test_roofline_fields_at_64_heads_count_the_flops_of_each_entry():
    entries = 128 * 2048
    r = bench.roofline_fields(64, entries * 1152.0, 1152, 0.1, PEAKS)
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s" and r["peak"] == 1700.0
    # each valid entry costs 64 heads x (576 + 512) multiply-adds
    assert r["achieved"] == pytest.approx(entries * 2 * 64 * 1088 / 0.1e-3 / 1e12)
    assert r["hbm_frac"] == pytest.approx(r["gathered_gbps"] / 6800.0)


def test_decode_batch_algorithmic_bytes():
    idx = torch.randint(0, 524288, (32, 2048), dtype=torch.int32)
    idx[0, :5] = -1
    idx[1, 0] = 524288  # out of range: masked, not gathered
    assert gathered_bytes(idx, 524288, 1152) == (32 * 2048 - 6) * 1152


def test_traffic_figures_are_used_only_for_their_kernel_sources(monkeypatch):
    d = json.loads((ROOT / "profiles" / "ncu_traffic.json").read_text())
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: d["kernel_source_hash"])
    got = bench.ncu_traffic("decode_bf16", 8, False)
    assert got == pytest.approx(d["entries"]["decode_bf16/h8"]["dram_bytes_per_launch"])
    # the decode launch reads each gathered row once: DRAM bytes within 10 % of 75.5 MB
    assert 1.0 <= got / (32 * 2048 * 1152) <= 1.1
    assert bench.ncu_traffic("decode_bf16", 8, True) is None  # no padded decode entry
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "0" * 16)
    assert bench.ncu_traffic("decode_bf16", 8, False) is None


def test_kernel_source_hash_covers_every_kernel_source(tmp_path, monkeypatch):
    src = tmp_path / "csrc"
    src.mkdir()
    (src / "a.cuh").write_text("x")
    (src / "b.cu").write_text("y")
    monkeypatch.setattr(bench, "CSRC", src)
    h0 = bench.kernel_source_hash()
    (src / "a.cuh").write_text("x ")
    assert bench.kernel_source_hash() != h0


def test_per_config_traffic_keys(monkeypatch):
    """The per-configuration entries look up traffic as (workload, heads launched, padded): the
    native sweep at 16 and 64 heads, the prefill chunk and the native fp8 batch have launch lists;
    padded arms have none of their own."""
    d = json.loads((ROOT / "profiles" / "ncu_traffic.json").read_text())
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: d["kernel_source_hash"])
    for name, h, h_real in (("sweep", 16, 16), ("sweep", 64, 64), ("prefill", 64, 64), ("fp8_mixed", 8, 8)):
        assert bench.ncu_traffic(name, h, h != h_real) is not None, (name, h)
    for name, h, h_real in (("sweep", 64, 8), ("fp8_mixed", 64, 8)):
        assert bench.ncu_traffic(name, h, h != h_real) is None, (name, h)
