"""The benchmark's launch-timeline summary (host logic, no GPU): interval unions, the
link's busy time, and the layer boundary measured between one layer's last page
read and the next layer's first, on hand-made launch records."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


T0 = 5_000_000  # device clock of the first launch, us (a record with start 0 never ran)


def rec(kind, layer, s_us, e_us, pages=0):
    return {"kind": kind, "layer": layer, "stream": 0, "pages": pages,
            "start_ns": int((T0 + s_us) * 1000), "end_ns": int((T0 + e_us) * 1000)}


def test_union_merges_overlaps_and_keeps_gaps():
    assert bench._union([]) == 0
    assert bench._union([(0, 10), (5, 15), (20, 25)]) == 20
    assert bench._union([(20, 25), (0, 10), (10, 12)]) == 17  # touching intervals merge, order does not matter
    assert bench._clip([(0, 10), (20, 30)], 5, 25) == [(5, 10), (20, 25)]


def test_summary_of_two_layers():
    recs = [
        rec("fill", 0, 0, 10, 4), rec("read_ring", 0, 10, 15, 4), rec("fill", 0, 12, 22, 4),
        rec("read_ring", 0, 22, 27, 4), rec("read_resident", 0, 11, 20, 64),
        rec("fill", 1, 24, 34, 4),                      # the next layer's first chunk, copied during layer 0
        rec("combine", 0, 30, 33), rec("clear", 0, 34, 36), rec("append", 1, 34, 35), rec("qprep", 1, 36, 37),
        rec("read_ring", 1, 40, 45, 4), rec("read_resident", 1, 41, 50, 64),
        {"kind": "fill", "layer": 1, "stream": 1, "pages": 4, "start_ns": 0, "end_ns": 0},  # never ran
    ]
    t = bench.timeline_summary(recs, 2)
    assert t["step_us"] == 50
    assert t["refill_busy_us"] == 30 and t["refill_launches"] == 3   # [0,10], [12,22], [24,34]
    # boundary: layer 0's last read ends at 27, layer 1's first read starts at 40
    assert t["boundary_us_median"] == 13 and t["boundary_us_total"] == 13
    # refills run 27..34 of that boundary's 13 us
    assert abs(t["refill_busy_in_boundaries_frac"] - 7 / 13) < 1e-9
    k = t["boundary_kernels_us_median"]
    assert k["combine (layer l)"] == 3 and k["append (layer l+1)"] == 1 and k["qprep (layer l+1)"] == 1
    assert k["clear (layer l)"] == 2


def test_summary_of_nothing_is_none():
    assert bench.timeline_summary([], 4) is None
