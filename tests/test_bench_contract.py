"""Host-side pieces of the benchmark line: the reference arm reports the decode arm's config,
per-step spreads are percentiles of the per-step times, and the host record names the cores
the single-threaded oracle used."""
import numpy as np
import pytest

import bench


def test_reference_arm_reports_the_decode_config():
    ours = bench.decode_config(8, True, 1)
    assert ours["workload"].startswith("decode MoE layer T=8")
    assert ours["T"] == 8 and ours["d"] == 4096 and ours["E"] == 384 and ours["k"] == 6
    assert ours == bench.decode_config(8, True, 1)   # one definition serves both arms
    assert "Engram" not in bench.decode_config(8, False, 1)["workload"]


def test_spread_is_percentiles_in_us():
    ms = [0.100, 0.120, 0.110, 0.300, 0.105, 0.115, 0.108, 0.112, 0.111, 0.109]
    sp = bench.spread_us(ms)
    q = np.percentile(np.array(ms) * 1e3, [10, 50, 90])
    assert sp == {"p10": pytest.approx(q[0], abs=0.01), "p50": pytest.approx(q[1], abs=0.01),
                  "p90": pytest.approx(q[2], abs=0.01)}
    assert sp["p10"] <= sp["p50"] <= sp["p90"]


def test_host_record_counts_cores():
    h = bench.host_cpu()
    assert h["nproc"] >= 1
    assert h["used"] == f"1 of {h['nproc']} cores"
