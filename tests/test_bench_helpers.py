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


def _fake_layer():
    rng = np.random.default_rng(0)
    out = []
    for name, n, k in (("a", 512, 256), ("b", 128, 1024), ("c", 256, 512)):
        spec = SimpleNamespace(name=name, rows=n, cols=k)
        m = dict(codes=rng.integers(0, 16, size=(n, k), dtype=np.uint8),
                 scales=rng.integers(0, 1 << 14, size=(n, k // 256), dtype=np.uint16),
                 mins=rng.integers(0, 1 << 14, size=(n, k // 256), dtype=np.uint16),
                 x=rng.standard_normal((1, k)).astype(np.float32))
        out.append((spec, m))
    return out


def test_oracle_shares_deal_every_strip_once():
    mats = _fake_layer()
    target = 3 * 64 * 1024 * 2          # two 64-row strips' worth of weights per matrix
    one = bench.oracle_shares(mats, target, 1)[0]
    for n in (1, 3, 5, 64):
        shares = bench.oracle_shares(mats, target, n)
        assert 1 <= len(shares) <= n
        # per matrix, the strips dealt out are exactly the one-worker sample's rows
        for j, (spec, m) in enumerate(mats):
            got = np.concatenate([sub["codes"] for sh in shares for sub in sh
                                  if sub["x"] is m["x"]] or [np.zeros((0, spec.cols), np.uint8)])
            want = [sub["codes"] for sub in one if sub["x"] is m["x"]][0]
            rows = sorted(map(bytes, got))
            assert rows == sorted(map(bytes, want))
        loads = [sum(sub["codes"].size for sub in sh) for sh in shares]
        assert max(loads) - min(loads) <= 64 * max(s.cols for s, _ in mats)


def test_oracle_all_cores_runs_every_share():
    mats = _fake_layer()
    r = bench.oracle_all_cores(mats, 3 * 64 * 1024, steps=1, warmup=0, cores=2)
    assert r["cores"] == 2 and r["value"] > 0 and r["seconds_per_pass"] > 0
    assert r["weights"] == sum(min(s.rows, max(64, (64 * 1024 // s.cols) // 64 * 64)) * s.cols
                               for s, _ in mats)


def test_reference_arm_prints_one_json_line(monkeypatch, capsys):
    """bench.py --impl reference on a small stand-in layer: one JSON line with
    the contract's keys, the oracle on every host core and on one."""
    import json
    monkeypatch.setattr(bench, "layer_matrices", _fake_layer)
    monkeypatch.setenv("RANK", "0")
    args = SimpleNamespace(steps=2, warmup=1, gpus=1, impl="reference")
    assert bench.run_reference(args) == 0
    lines = [ln for ln in capsys.readouterr().out.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "GB/s"
    assert d["value"] > 0 and d["higher_is_better"] is True and d["steps"] == 2
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1
    assert cb["single_core"]["cores"] == 1 and cb["single_core"]["value"] > 0
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_reference_arm_other_ranks_do_nothing(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setattr(bench, "layer_matrices", lambda: (_ for _ in ()).throw(AssertionError))
    assert bench.run_reference(SimpleNamespace(steps=2, warmup=1, gpus=2, impl="reference")) == 0
    assert capsys.readouterr().out == ""


def test_reference_arm_falls_back_to_one_core(monkeypatch, capsys):
    import json

    def broken(*a, **k):
        raise RuntimeError("no workers")
    monkeypatch.setattr(bench, "layer_matrices", _fake_layer)
    monkeypatch.setattr(bench, "oracle_all_cores", broken)
    monkeypatch.setenv("RANK", "0")
    assert bench.run_reference(SimpleNamespace(steps=1, warmup=0, gpus=1, impl="reference")) == 0
    d = json.loads(capsys.readouterr().out.strip())
    assert d["cpu_baseline"]["cores"] == 1 and d["value"] == d["cpu_baseline"]["single_core"]["value"]
    assert "unavailable: no workers" in d["cpu_baseline"]["sample"]


class _FakeCuda:
    """Just enough of torch.cuda for bench's timing helpers on the CPU: events
    read a counter that every step advances by the step's index + 1 ms."""

    def __init__(self):
        self.now = 0.0

    def Event(self, enable_timing=True):
        cuda = self

        class E:
            def record(self, stream=None):
                self.t = cuda.now

            def elapsed_time(self, other):
                return other.t - self.t
        return E()

    def synchronize(self):
        pass

    def CUDAGraph(self):
        return SimpleNamespace(replay=lambda: None)

    def graph(self, g):
        import contextlib
        return contextlib.nullcontext()


def test_timing_helpers_with_a_fake_device():
    cuda = _FakeCuda()
    torch = SimpleNamespace(cuda=cuda)
    seen = []

    def step(c):
        seen.append(c)
        cuda.now += 1.0 + c          # copy c takes c + 1 ms
    # mean over steps rotating over 3 copies: (1 + 2 + 3) / 3
    assert bench.time_steps(torch, None, step, steps=6, warmup=2, copies=3) == 2.0
    assert seen[:2] == [0, 1] and seen[2:] == [0, 1, 2, 0, 1, 2]
    ms = bench.per_step_ms(torch, None, step, steps=4, copies=2)
    assert ms == [1.0, 2.0, 1.0, 2.0]
    sp = bench.percentiles(ms)
    assert sp["median"] == 1.5 and sp["steps"] == 4
    # a layer graph: the calls run once eagerly, then once more, in order,
    # under the capture
    calls = []
    bench.layer_graph(torch, [lambda: calls.append("a"), lambda: calls.append("b")])
    assert calls == ["a", "b", "a", "b"]
