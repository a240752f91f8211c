"""The benchmark's JSON line (no GPU): the keys the measurement contract asks
for, and the arithmetic of value, e2e and the roofline from given durations."""
import json

import bench

GB = 1e9


def _args(**kw):
    class A:
        pass

    a = A()
    a.type, a.steps, a.warmup, a.layers, a.n_kv = "q8_0", 500, 5, 64, 16384
    for k, v in kw.items():
        setattr(a, k, v)
    return a


def test_step_line_keys_and_arithmetic():
    a = _args()
    L, n = 64, 16384
    # 0.9 ms per step, 14 us per attention launch, e2e 0.94 ms, two calls 1.03 ms
    line = bench.step_line(a, 1, L, n, 0.9e-3 * 500, 14e-6 * 64 * 500, 0.94e-3 * 500, 1.03e-3 * 500,
                           1835008, 1310720, {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": []})
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "roofline", "e2e", "gpu_launches", "clocks"):
        assert k in line, k
    json.dumps(line)
    step_bytes = L * n * 2176
    assert abs(line["value"] - step_bytes / 0.9e-3 / GB) < 0.01
    assert line["ms_per_step"] == 0.9 and line["steps"] == 500 and line["warmup"] == 5
    assert line["higher_is_better"] is True and line["scaling"] == "weak" and line["vs_baseline"] is None
    assert line["gpu_launches"] == L * 500
    r = line["roofline"]
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert abs(r["achieved"] - n * 2176 / 14e-6 / GB) < 0.1 and abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-4
    assert abs(line["e2e"]["value"] - step_bytes / 0.94e-3 / GB) < 0.01
    assert line["e2e"]["h2d_bytes_per_step"] == 1835008 and line["e2e"]["d2h_bytes_per_step"] == 1310720
    assert line["config"]["workload"].startswith("decode, 64 layers")


def test_value_is_whole_job_over_ranks():
    a = _args()
    one = bench.step_line(a, 1, 64, 16384, 0.45, 0.448, 0.47, 0.52, 1, 1, {})
    two = bench.step_line(a, 2, 64, 16384, 0.45, 0.448, 0.47, 0.52, 1, 1, {})
    assert abs(two["value"] - 2 * one["value"]) < 0.02 and two["n_gpus"] == 2
    assert abs(two["hbm_frac"] - one["hbm_frac"]) < 1e-4  # per-GPU fraction


def test_timeline_summary_of_a_constructed_trace():
    # two layers, three steps; each layer: a 1 MB delivery of 10 us, then a 5 us attention that
    # overlaps the next layer's delivery by 2 us
    recs, t = [], 0.0
    for _ in range(3):
        for l in range(2):
            recs.append((0, l, 1_000_000, t, t + 10.0))
            recs.append((1, l, 0, t + 10.0, t + 15.0))
            t += 13.0
    s = bench.timeline_summary(recs, 2)
    assert s["step_ms"] == 0.026 and s["deliveries"] == 2
    assert s["per_delivery_gbs_p10_p50_p90"] == [100.0, 100.0, 100.0]
    # per step (26 us): copies busy 20 us, attention 10 us, 2 x 2 us of copy hidden
    assert s["copy_busy_frac"] == round(20 / 26, 3) and s["attn_busy_frac"] == round(10 / 26, 3)
    assert s["copy_hidden_frac"] == round(4 / 20, 3) and s["attn_hidden_frac"] == round(4 / 10, 3)
    assert s["launches_per_step"] == 2
    assert "error" in bench.timeline_summary(recs[:4], 2)
    # rolling tiles: two attention launches per layer, the step found from the launch count
    recs2, t = [], 0.0
    for _ in range(3):
        for l in range(2):
            for _tile in range(2):
                recs2.append((0, l, 500_000, t, t + 5.0))
                recs2.append((1, l, 0, t + 5.0, t + 7.0))
                t += 7.0
    s2 = bench.timeline_summary(recs2, 2)
    assert s2["launches_per_step"] == 4 and s2["step_ms"] == 0.028 and s2["deliveries"] == 4


def test_clock_summary_keeps_the_samples_inside_the_timed_windows():
    import datetime

    def line(ts, sm, reasons=("Not Active",) * 4):
        stamp = datetime.datetime.fromtimestamp(ts).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
        return "%s, 0, %d, 2070, 900.5, 0x0, %s" % (stamp, sm, ", ".join(reasons))

    t0 = 1_800_000_000.0
    lines = [line(t0 - 1.0, 900), line(t0 + 0.1, 2070), line(t0 + 0.2, 2060),
             line(t0 + 0.3, 2070, ("Not Active", "Not Active", "Not Active", "Active")),
             line(t0 + 5.0, 1200), "garbage line"]
    got = bench.clock_summary(lines, [(t0, t0 + 0.35)])
    assert got["samples"] == 3 and got["sm_mhz"] == 2070.0 and got["sm_max_mhz"] == 2070.0
    assert got["reasons"] == ["sw_power_cap"] and got["note"].startswith("samples inside")
    # a window with no sample inside reports the nearest sample, and says so
    got = bench.clock_summary(lines, [(t0 + 4.0, t0 + 4.01)])
    assert got["samples"] == 1 and got["sm_mhz"] == 1200.0 and got["note"].startswith("no sample")
    assert bench.clock_summary([], [(t0, t0 + 1)])["sm_mhz"] is None
