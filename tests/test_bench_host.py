"""Host-side logic of bench.py (CPU): the FLOP counts against the workloads'
figures worked out by hand, and the clock-record summary."""
import os
import sys
import time

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_flop_counts():
    # LayerNormMLP fwd+bwd: six GEMMs of 2*M*D*F each
    assert bench.flops_per_step(8192, 768, 3072) == 6 * 2 * 8192 * 768 * 3072
    assert abs(bench.flops_per_step() / 1e9 - 231.928) < 1e-3
    # one transformer-block layer at d 2048 over 16384 tokens: QKV 1236.9, projection 412.3, MLP 3298.5 GFLOP
    per_layer = bench.stack_flops_per_step(1, 16384, 2048, 8192) / 1e9
    assert abs(per_layer - (1236.95 + 412.32 + 3298.53)) < 0.05
    assert abs(bench.stack_flops_per_step(12, 16384, 2048, 8192) / 1e12 - 59.38) < 0.01


def _line(ts, sm, reasons=("Not Active",) * 4):
    return ", ".join([ts, "0", str(sm), "2070", "500.0", "0x0"] + list(reasons)) + "\n"


def test_clock_summary_keeps_samples_inside_the_region():
    base = time.mktime(time.strptime("2026/12/02 10:00:00", "%Y/%m/%d %H:%M:%S"))
    lines = [_line("2026/12/02 10:00:00.000", 1000),                      # before the region
             _line("2026/12/02 10:00:01.000", 2070),
             _line("2026/12/02 10:00:01.500", 2000, ("Not Active", "Not Active", "Not Active", "Active")),
             _line("2026/12/02 10:00:02.000", 1900),
             _line("2026/12/02 10:00:05.000", 500),                       # after it
             "garbage line\n"]
    out = bench.ClockSampler.summarize(lines, base + 0.9, base + 2.1)
    assert out["samples"] == 3 and out["sm_mhz"] == 2000 and out["sm_max_mhz"] == 2070
    assert out["reasons"] == ["sw_power_cap"]
    everything = bench.ClockSampler.summarize(lines)
    assert everything["samples"] == 5 and everything["sm_mhz"] == 1900
    assert bench.ClockSampler.summarize([])["sm_mhz"] is None


def test_stack_hbm_bytes_by_hand():
    # one layer at d 2048 over 16384 tokens: the QKV LayerNorm reads x (2 B) and writes codes (1 B),
    # the MLP LayerNorm adds the residual (x, r read, h written, codes: 7 B); 8 B of mu, rsigma per row;
    # the QKV LayerNorm launch also casts the QKV weight (6144 x 2048, below 2^24 elements: 2 B read,
    # 1 B written); W1 and W2 (8192 x 2048 = 2^24 each) stream through their own cast launches
    md = 16384 * 2048
    b = bench.stack_hbm_bytes(1, 16384, 2048, 8192)
    assert b["ln_fwd_cast"] == 3 * md + 7 * md + 2 * 8 * 16384 + 3 * 3 * 2048 * 2048
    assert b["ln_bwd"] == 2 * (6 * md + 8 * 16384)
    assert b["cast_colsum"] == 3 * 5 * md + 4 * 5 * 2048         # dY of MLP and projection, dQKV (3d wide)
    assert b["cast"] == 3 * 2048 * 2048 + 3 * md + 3 * 2 * 8192 * 2048  # projection weight and input, W1, W2
    assert "cast_pair" not in b
    twelve = bench.stack_hbm_bytes(12, 16384, 2048, 8192)
    assert twelve["ln_fwd_cast"] == 3 * md + 23 * 7 * md + 24 * 8 * 16384 + 12 * 3 * 3 * 2048 * 2048
    # at d 768 every weight rides in a LayerNorm launch
    s768 = bench.stack_hbm_bytes(4, 8192, 768, 3072)
    assert s768["ln_fwd_cast"] == 3 * 8192 * 768 + 7 * 7 * 8192 * 768 + 8 * 8 * 8192 + 4 * 3 * (3 * 768 * 768 + 2 * 3072 * 768)
    assert s768["cast"] == 4 * (3 * 768 * 768 + 3 * 8192 * 768)
