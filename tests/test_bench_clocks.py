"""The bench's clock record keeps only nvidia-smi samples taken inside the
timed region (host logic, no GPU)."""
import datetime
import os
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _sampler_with(rows, t0, t1):
    c = bench.ClockSampler(0)
    fd, c.path = tempfile.mkstemp(suffix=".csv")
    os.close(fd)
    with open(c.path, "w") as f:
        for t, mhz, watts, cap in rows:
            ts = datetime.datetime.fromtimestamp(t).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
            f.write(f"{ts}, {mhz}, 2070, {watts}, 0x0, Not Active, Not Active, Not Active, "
                    f"{'Active' if cap else 'Not Active'}\n")
    c.proc = object()  # summary() only checks that a sampler ran
    c.t0, c.t1 = t0, t1
    return c


def test_only_samples_inside_the_timed_region_count():
    now = time.time()
    rows = [(now - 0.5, 2070, 200, False), (now + 0.1, 1800, 1300, False),
            (now + 0.2, 1750, 1390, True), (now + 0.9, 2070, 220, False)]
    s = _sampler_with(rows, now, now + 0.5).summary()
    assert s["samples"] == 2 and s["samples_total"] == 4
    assert s["sm_mhz"] == 1775.0
    assert s["reasons"] == ["sw_power_cap"]
    assert s["window"] == "samples inside the timed region"


def test_falls_back_to_all_samples_when_none_is_inside():
    now = time.time()
    rows = [(now - 0.5, 2070, 200, False), (now + 2.0, 1900, 900, False)]
    s = _sampler_with(rows, now, now + 0.1).summary()
    assert s["samples"] == 2
    assert s["window"].startswith("all samples")
