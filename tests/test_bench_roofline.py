"""bench.py's roofline arithmetic against closed forms (CPU): entry sizes of both formats, the
decode expert kernel's achieved bandwidth on calls without misses, and the step figure that
adds the routing time and the router weights."""
import math

import bench


def test_entry_bytes_both_formats():
    wl = dict(bench.WORKLOADS["decode24"])
    assert bench.entry_bytes(wl) == 3 * 2048 * 768 * 2 == 9_437_184
    wl["fp4"] = True
    # codes: 4 bits per weight; scales: one byte per 32 weights -> 17/32 byte per weight
    assert bench.entry_bytes(wl) == 3 * 2048 * 768 // 2 + 3 * 2048 * 768 // 32
    wl8 = dict(bench.WORKLOADS["large8"])
    assert bench.entry_bytes(wl8) == 3 * 4096 * 2048 * 2


def test_roofline_decode_closed_forms():
    wl = dict(bench.WORKLOADS["decode24"])
    eb = 9_437_184
    # 10 launches without misses streaming 80 entries in 0.35 ms, 14 with misses, 24 routing
    # launches in 0.39 ms
    prof = {"experts_hit": (0.35, 10, 80), "experts_miss": (3.7, 14, 112),
            "router": (0.39, 24, 0)}
    rl = bench.roofline_decode(wl, prof, bench.peaks())
    hit = rl["experts_hit"]
    assert hit["bytes"] == 80 * eb
    assert math.isclose(hit["achieved"], 80 * eb / 0.35e-3 / 1e9, rel_tol=1e-12)
    assert rl["experts_miss"]["hbm_bytes"] == 112 * eb
    route = 0.39 / 24
    assert math.isclose(rl["route_us_per_call"], route * 1e3, rel_tol=1e-12)
    m2 = rl["step_m2"]
    assert m2["bytes"] == 80 * eb + 10 * 128 * 2048 * 2
    assert math.isclose(m2["ms"], 0.35 + route * 10, rel_tol=1e-12)
    assert math.isclose(m2["achieved"], m2["bytes"] / (m2["ms"] / 1e3) / 1e9, rel_tol=1e-12)


def test_roofline_decode_no_launches_is_zero():
    wl = dict(bench.WORKLOADS["decode24"])
    prof = {"experts_hit": (0.0, 0, 0), "experts_miss": (0.0, 0, 0), "router": (0.0, 0, 0)}
    rl = bench.roofline_decode(wl, prof, bench.peaks())
    assert rl["experts_hit"]["achieved"] == 0.0 and rl["step_m2"]["achieved"] == 0.0
    assert rl["route_us_per_call"] == 0.0
