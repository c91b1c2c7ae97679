"""bench.py on the CPU: the reference arm's JSON line, the roofline arithmetic, the traffic table lookup."""

import contextlib
import io
import json
import os

import pytest

import bench


def test_reference_arm_prints_the_contract_line():
    out = io.StringIO()
    with contextlib.redirect_stdout(out):
        rc = bench.main(["--impl", "reference", "--steps", "2", "--warmup", "3"])
    assert rc == 0
    line = json.loads(out.getvalue().strip().splitlines()[-1])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in line, k
    assert line["impl"] == "reference" and line["value"] > 0 and line["steps"] == 2 and line["warmup"] == 3
    assert line["metric"] == bench.METRIC and line["unit"] == "tokens/s" and line["higher_is_better"] is True
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    assert line["config"]["workload"].startswith("adapter4k")


class _Wl:
    def __init__(self, bound, b, f):
        self.bound, self.bytes_per_call, self.flops_per_call = bound, b, f


def test_roofline_object_arithmetic():
    peaks = {"hbm_gbs": 6000.0, "bf16_tflops": 1500.0, "bf16_tflops_sustained": 1200.0}
    r = bench.roofline_obj(_Wl("hbm", 3e6, 1e9), 0.01, peaks, 12345)      # 3 MB in 10 us = 300 GB/s
    assert r["unit"] == "GB/s" and abs(r["achieved"] - 300.0) < 1e-6 and abs(r["frac"] - 0.05) < 1e-9
    assert r["traffic"] == 12345
    r = bench.roofline_obj(_Wl("tensor", 1e6, 7.5e11), 1.0, peaks, None)  # 7.5e11 FLOP in 1 ms = 750 TF/s
    assert r["unit"] == "TFLOP/s" and abs(r["achieved"] - 750.0) < 1e-6
    assert abs(r["frac"] - 0.5) < 1e-9 and abs(r["frac_of_sustained"] - 0.625) < 1e-9


def test_traffic_table_entries_name_existing_sources_and_go_stale_when_they_change(monkeypatch, tmp_path):
    table = json.load(open(os.path.join(bench.ROOT, "profiles", "dram_traffic.json")))
    for key, e in table.items():
        if key == "about":
            continue
        for f in e["sources"]:
            assert os.path.exists(os.path.join(bench.ROOT, "double_binary_rank_packed_b300", "csrc", f)), f
        assert e["dram_bytes_per_launch"] > 0
    # a table whose hash does not match the sources reads as unknown traffic
    key = next(k for k in table if k != "about")
    stale = dict(table)
    stale[key] = dict(table[key], sources_hash="0" * 16)
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "dram_traffic.json").write_text(json.dumps(stale))
    (tmp_path / "double_binary_rank_packed_b300").symlink_to(os.path.join(bench.ROOT, "double_binary_rank_packed_b300"))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.measured_traffic(key) is None
    assert bench.measured_traffic("no_such_workload") is None


@pytest.mark.parametrize("key", bench.SECONDARY)
def test_every_secondary_workload_has_a_title(key):
    if "_T" not in key:   # not a token workload (the factorization round)
        assert key in bench.WORKLOAD_TITLES
        return
    name, _, tok = key.rpartition("_T")
    assert name in bench.WORKLOAD_TITLES and int(tok) > 0


def test_factorize_flop_count():
    # one step at N = M = 4096, k = 3072, 10 iterations: F F^T 77.3 G, T F^T 103.1 G,
    # inverse 29.0 G, ten P-updates 773.1 G
    f = bench.factorize_step_flops(4096, 4096, 3072, 10)
    assert abs(f - (2 * 3072 ** 2 * 4096 + 2 * 4096 * 3072 * 4096 + 3072 ** 3 + 10 * 2 * 4096 * 3072 ** 2)) == 0
    assert 0.98e12 < f < 0.99e12


def test_alu_roofline():
    class W:
        bound, flops_per_call, alu_peak_tflops = "alu", 2e12, 77.0
    r = bench.roofline_obj(W(), 50.0, None, None)     # 2 TFLOP in 50 ms = 40 TF/s
    assert r["unit"] == "TFLOP/s" and abs(r["achieved"] - 40.0) < 1e-9 and abs(r["frac"] - 40 / 77) < 1e-4
