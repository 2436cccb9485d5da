"""bench.py's host-side helpers (no GPU): how a step's matrices are grouped
into launches, and the byte count of a tile-skip launch list."""
from types import SimpleNamespace

import numpy as np

import bench
from decode_gemv_gb300 import inputs
from decode_gemv_gb300 import lw


def test_layer_groups():
    names = ["q", "k", "v", "o", "gate", "up", "down"]
    assert bench.layer_groups(names) == [[0, 1, 2], [3], [4, 5], [6]]
    assert bench.layer_groups(names, ungrouped=True) == [[i] for i in range(7)]
    assert bench.layer_groups(["gate", "down"]) == [[0], [1]]
    assert bench.layer_groups(["v", "q"]) == [[1, 0]]          # layer order within a group


def test_sweep_groups_per_layer_and_format():
    S = lambda n: SimpleNamespace(name=n)
    L = SimpleNamespace(LW_FMT_BF16_EXP=lw.LW_FMT_BF16_EXP)
    q4, bf = lw.LW_FMT_Q4_PAIR, lw.LW_FMT_BF16_EXP
    mats = [dict(spec=S(n), fmt=f, layer=l) for l in range(2)
            for n, f in [("q", q4), ("k", q4), ("v", q4), ("o", q4), ("gate", bf), ("up", bf), ("down", bf)]]
    g = bench.sweep_groups(mats, L)
    assert g == [[0, 1, 2], [3], [4], [5], [6], [7, 8, 9], [10], [11], [12], [13]]
    # every matrix exactly once
    assert sorted(i for grp in g for i in grp) == list(range(len(mats)))
    mats = [dict(spec=S(n), fmt=q4, layer=0) for n in ["qkv", "o", "gate_up", "down"]]
    assert bench.sweep_groups(mats, L) == [[0], [1], [2], [3]]


def test_listed_bytes_counts_the_listed_tiles():
    n, k = 256, 1024
    m = inputs.small_q4(3, n, k)
    hb = lw.lw_encode_bundle(lw.LW_FMT_Q4_PAIR, m["codes"], m["scales"], m["mins"])
    tk, strips = k // 256, n // 64
    secs = hb.sections
    # all strips: every section's bytes (the table once)
    full = bench.listed_bytes(hb, list(range(strips)), k)
    assert full == sum(len(v) for v in secs.values())
    # the listed strips' words plus their per-tile side data
    toff = hb.view("tile_off", np.uint32).astype(np.int64)
    for lst, n_off in (([0], tk + 1), ([1, 3], 2 * (tk + 1)), ([1, 2], 2 * tk + 1)):
        words = sum(int(toff[(s + 1) * tk] - toff[s * tk]) * 128 for s in lst)
        per_tile = 64 + 64 + 256          # lane bits, lane mids, scales/mins
        assert bench.listed_bytes(hb, lst, k) == words + len(lst) * tk * per_tile + 4 * n_off + 1024


def test_percentiles_of_step_times():
    # 1..101 ms: the order statistics fall on whole values
    s = bench.percentiles(np.arange(1, 102, dtype=np.float64)[::-1])
    assert s == {"p10": 11.0, "median": 51.0, "p90": 91.0, "steps": 101}
    one = bench.percentiles([0.25])
    assert one["p10"] == one["median"] == one["p90"] == 0.25 and one["steps"] == 1
