"""The trace tool's page-issue summary on a hand-built trace (no GPU): the idle
time and the issue rate of a layer are fixed by the timestamps written here."""
import numpy as np
import pytest

from decode_megakernel_persistent_gb300 import trace


def hand_trace():
    # two SMs, three layers of the five matrix/attention instructions each
    nsm, L = 2, 3
    plan = np.full((nsm, 5 * L + 1, 7), -1, dtype=np.int32)
    tr = np.zeros((nsm, 5 * L + 1, 12), dtype=np.int64)
    for sm in range(nsm):
        for l in range(L):
            for k in range(5):
                i = 5 * l + k
                plan[sm, i, 0], plan[sm, i, 1] = k, l
                tr[sm, i, 0] = l * 10_000 + k * 2_000           # begin, ns
                tr[sm, i, 3] = l * 10_000 + (k + 1) * 2_000 - (500 if sm else 0)  # end
    # layer 1 runs from 10 us (layer 0's down ends on SM 0) to 20 us; each SM
    # issues a page every 100 ns from 10.0 to 14.9 us, then none
    pt = np.zeros((nsm, 64, 3), dtype=np.int64)
    for sm in range(nsm):
        pt[sm, :50, 0] = 10_000 + 100 * np.arange(50)
    return tr, pt, plan


def test_issue_idle_closed_form():
    tr, pt, plan = hand_trace()
    r = trace.issue_idle(tr, pt, plan, bin_us=0.5, idle_pages=5)
    assert r["layer_span_us"] == pytest.approx(10.0)
    assert r["idle_us"] == pytest.approx(5.0)  # 15-20 us: nothing issued
    # 10 pages (both SMs) per 0.5 us bin
    assert r["busy_issue_gbs"] == pytest.approx(10 * 32768 / 0.5e-6 / 1e9, rel=1e-3)


def test_issue_idle_threshold():
    tr, pt, plan = hand_trace()
    # with 10 pages a bin counted as idle, the whole layer is idle
    r = trace.issue_idle(tr, pt, plan, bin_us=0.5, idle_pages=10)
    assert r["idle_us"] == pytest.approx(10.0)
    assert r["busy_issue_gbs"] == 0.0
