"""Host-side numbers of bench.py from synthetic loop records (no GPU): the headline
divides steps by the summed step times, miss and hit steps are reported apart, the
per-launch kernel time comes only from records that carry kernel brackets, and the
committed ncu traffic line is well formed."""
from types import SimpleNamespace

import bench


def _bench(layers=1, batch=1):
    return SimpleNamespace(sp=SimpleNamespace(layers=layers, batch=batch))


def _rec(ms, miss, kernel_ms=None, scan=268_435_456, gather=10_500_000):
    prof = {} if kernel_ms is None else {"step": (kernel_ms, 1), "score": (0.0, 0)}
    return dict(t=0, ms=ms, prof=prof, any_miss=miss, n_miss=int(miss), scan=scan if miss else 0, gather=gather)


def test_headline_and_split_by_hits():
    rec = [_rec(0.120, True), _rec(0.030, False), _rec(0.122, True), _rec(0.032, False)]
    s = bench.summarise(_bench(), rec, 6668.5)
    total = 0.120 + 0.030 + 0.122 + 0.032
    assert abs(s["ms_per_step"] - total / 4) < 1e-12
    assert abs(s["value"] - 4000.0 / total) < 1e-9
    assert abs(s["miss_ms_per_step"] - 0.121) < 1e-12
    assert abs(s["hit_ms_per_step"] - 0.031) < 1e-12
    assert abs(s["hit_rate"] - 0.5) < 1e-12
    assert "score_us_per_launch" not in s            # no kernel brackets in these records


def test_kernel_time_from_bracketed_records():
    rec = [_rec(0.125, True, kernel_ms=0.120), _rec(0.031, False, kernel_ms=0.023), _rec(0.127, True, kernel_ms=0.122)]
    s = bench.summarise(_bench(), rec, 6668.5)
    assert s["fused"]
    assert abs(s["score_us_per_launch"] - 121.0) < 1e-9          # miss launches only
    bytes_per = 268_435_456 + 10_500_000
    assert abs(s["scan_bytes_per_launch"] - bytes_per) < 1e-6
    assert abs(s["score_gbs"] - 2 * bytes_per / (0.242e-3) / 1e9) < 1e-6


def test_timed_takes_step_numbers_and_kernel_numbers_from_their_loops():
    class FakeBench:
        sp = SimpleNamespace(layers=1, batch=1, steps=4)

        def run(self, steps, warmup, flush=True):
            return [_rec(0.200, True, kernel_ms=0.120) for _ in range(steps)]

        def run_async(self, steps, warmup, flush=True):
            return [_rec(0.125, True) for _ in range(steps)]

    s = bench.timed(FakeBench(), 4, 3, 6668.5)
    assert abs(s["ms_per_step"] - 0.125) < 1e-12                   # the back-to-back loop
    assert abs(s["score_us_per_launch"] - 120.0) < 1e-9            # the synchronised loop's brackets


def test_committed_traffic_line_is_well_formed():
    # (the bench uses it only while its source digest matches; that is checked at run time)
    import os
    import re
    text = "".join(open(os.path.join(bench.ROOT, "profiles", f)).read()
                   for f in os.listdir(os.path.join(bench.ROOT, "profiles")) if f.endswith(".md"))
    m = re.search(r"step_traffic_bytes_per_launch_n128k:\s*([0-9.e+]+)\s+step_source_sha256:\s*([0-9a-f]{64})", text)
    assert m is not None
    assert 270e6 < float(m.group(1)) < 300e6                       # ~K scan + gathers + small writes


def test_minimum_bytes_count_the_scan_and_the_selected_v_rows():
    # the algorithmic bytes count K and V of every selected token; the minimum counts the K scan
    # and the V rows only (the range attention reuses the scan's logits and reads no K row again)
    rec = [_rec(1.0, True, scan=2_147_483_648, gather=3_600_000_000), _rec(1.0, False, gather=3_600_000_000)]
    s = bench.summarise(_bench(), rec, 6668.5)
    alg = 2_147_483_648 + 2 * 3_600_000_000
    low = 2_147_483_648 + 2 * 1_800_000_000
    assert abs(s["step_gbs"] - alg / 2e-3 / 1e9) < 1e-6
    assert abs(s["min_step_gbs"] - low / 2e-3 / 1e9) < 1e-6
    assert abs(s["min_frac_of_peak"] - s["min_step_gbs"] / 6668.5) < 1e-12
    assert s["min_step_gbs"] < s["step_gbs"]


def test_cpu_model_is_named():
    assert isinstance(bench.cpu_model(), str) and bench.cpu_model()
