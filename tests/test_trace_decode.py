"""Decoding and summarising timeline records (no GPU)."""
import json

import numpy as np

from all_gather_gemm_gb300 import trace


def _buf(records, cap):
    b = np.zeros(1 + 4 * cap, np.uint64)
    b[0] = len(records)
    for i, (t0, t1, role, cta, a, bb) in enumerate(records[:cap]):
        b[1 + 4 * i:5 + 4 * i] = [t0, t1, (role << 56) | (cta << 40) | (a << 20) | bb, 0]
    return b


def test_decode_fields_and_relative_times():
    recs = [(1000, 1500, 2, 3, 17, 5), (900, 950, 1, 0, 2, 7), (2000, 9000, 3, 151, 127, 13)]
    d = trace.decode(_buf(recs, 8))
    assert d["count"] == 3 and d["dropped"] == 0
    assert list(d["start"]) == [100, 0, 1100] and list(d["end"]) == [600, 50, 8100]
    assert list(d["role"]) == [2, 1, 3] and list(d["cta"]) == [3, 0, 151]
    assert list(d["a"]) == [17, 2, 127] and list(d["b"]) == [5, 7, 13]


def test_overflowing_records_are_counted_as_dropped():
    recs = [(i, i + 1, 3, 0, 0, 0) for i in range(10)]
    d = trace.decode(_buf(recs, 4))
    assert d["count"] == 10 and d["dropped"] == 6 and d["start"].size == 4


def test_summary_and_chrome_json(tmp_path):
    recs = [(0, 2000, 2, 0, 1, 0), (0, 1000, 2, 1, 1, 0), (5000, 6000, 2, 0, 2, 0),
            (0, 0, 1, 1, 1, 0), (1000, 30000, 3, 0, 1, 0),
            (0, 400, 6, 0, 1, 0), (400, 1400, 6, 0, 1, 1 << 16)]
    d = trace.decode(_buf(recs, 16))
    s = trace.summarize(d, num_ctas=2)
    assert s["wait"]["n"] == 3
    assert abs(s["wait"]["per_cta_total_us_max"] - 3.0) < 1e-9   # CTA 0: 2 us + 1 us
    assert abs(s["wait"]["per_cta_total_us_mean"] - 2.0) < 1e-9
    assert abs(s["tile"]["done_by_us"]["p100"] - 30.0) < 1e-9
    assert s["issue"]["mean_us_by_kind"] == {"follower": 0.4, "local": 1.0}
    p = tmp_path / "t.json"
    trace.to_chrome_json(d, str(p))
    ev = json.load(open(p))["traceEvents"]
    assert len(ev) == len(recs) and {e["tid"] for e in ev} == {0, 1}
