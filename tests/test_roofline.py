"""The bench's roofline helper against the worked example of "MTP in
llama.cpp", section "Theoretical maximum tg t/s" (tests/golden/roofline_habr.txt)."""
from pathlib import Path

import pytest

import bench

GOLDEN = Path(__file__).resolve().parent / "golden" / "roofline_habr.txt"


def _golden():
    vals = {}
    for line in GOLDEN.read_text().splitlines():
        if line and not line.startswith("#"):
            k, v = line.split()
            vals[k] = float(v)
    return vals


def test_worked_example_bound():
    g = _golden()
    gib = 1 << 30
    bound = bench.roofline_rate(g["bandwidth_gib_s"] * gib, g["weights_gib"] * gib)
    # 268 / 13.5 = 19.85; the page writes 19.8 (one decimal, truncated)
    assert int(bound * 10) / 10 == g["bound_tokens_per_s"]
    assert g["measured_tokens_per_s"] / bound == pytest.approx(0.862, abs=0.005)


def test_bound_scales_inversely_with_bytes():
    assert bench.roofline_rate(6.6517e12, 14.17e9) == pytest.approx(469.4, rel=1e-3)
    assert bench.roofline_rate(2.0, 1.0) == 2 * bench.roofline_rate(1.0, 1.0)
