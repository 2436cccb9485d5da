"""One launch for several independent 4-/6-bit matrices
(lw_decode_gemv_group): every output bitwise equal to its matrix's own
lw_decode_gemv call and within tolerance of the oracle; matrices of different
shapes, tables and tile sizes in one group; shared inputs; argument errors."""
import numpy as np
import pytest

import oracle
from decode_gemv_gb300 import inputs
from decode_gemv_gb300 import lw
from helpers import assert_close

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lw.load()


def _mat(fmt, seed, n, k, sd=1.6):
    return inputs.small_q4(seed, n, k, sd=sd) if fmt == lw.LW_FMT_Q4_PAIR else inputs.small_q6(seed, n, k)


def _upload(fmt, m):
    hb = lw.lw_encode_bundle(fmt, m["codes"], m["scales"], m.get("mins"))
    return lw.DeviceBundle.upload(hb, DEV)


def _single(db, x):
    y = torch.full((db.rows,), float("nan"), device=DEV)
    ws = torch.zeros(lw.lw_workspace_bytes(db, 1) // 4 + 64, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    lw.lw_decode_gemv(db, x, y, ws, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return y.cpu().numpy()


SHAPES = [(1024, 4096), (64, 256), (256, 1024), (192, 3072), (512, 512), (320, 768), (128, 2048),
          (64, 1024)]


@pytest.mark.parametrize("fmt", [lw.LW_FMT_Q4_PAIR, lw.LW_FMT_Q6])
@pytest.mark.parametrize("n", [1, 3, 8])
def test_group_equals_single_calls(fmt, n):
    mats = [_mat(fmt, 100 * n + i, *SHAPES[i], sd=1.2 + 0.15 * i) for i in range(n)]
    dbs = [_upload(fmt, m) for m in mats]
    xs = [torch.from_numpy(m["x"][0]).to(DEV) for m in mats]
    ys = [torch.full((d.rows,), float("nan"), device=DEV) for d in dbs]
    ws = torch.zeros(lw.lw_workspace_bytes_group(dbs) // 4 + 64, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    for _ in range(2):   # twice: the counters are left at zero
        lw.lw_decode_gemv_group(dbs, xs, ys, ws, st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        for m, d, x, y in zip(mats, dbs, xs, ys):
            yg = y.cpu().numpy()
            assert np.array_equal(yg.view(np.uint32), _single(d, x).view(np.uint32))
            assert_close(yg[None], oracle.reference_output(fmt, m), oracle.abs_row_products(fmt, m))


def test_group_of_a_layer_with_shared_input():
    """q, k, v of a Mistral-shaped layer (full size) reading one x."""
    specs = inputs.workload_specs(inputs.MISTRAL_LAYER)[:3]
    mats = [inputs.make_matrix(inputs.MISTRAL_LAYER, s, 0, i) for i, s in enumerate(specs)]
    dbs = [_upload(lw.LW_FMT_Q4_PAIR, m) for m in mats]
    x = torch.from_numpy(mats[0]["x"][0]).to(DEV)
    ys = [torch.empty(d.rows, device=DEV) for d in dbs]
    ws = torch.zeros(lw.lw_workspace_bytes_group(dbs) // 4 + 64, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    lw.lw_decode_gemv_group(dbs, [x, x, x], ys, ws, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for d, y in zip(dbs, ys):
        assert np.array_equal(y.cpu().numpy().view(np.uint32), _single(d, x).view(np.uint32))


def test_group_argument_errors():
    m4 = _mat(lw.LW_FMT_Q4_PAIR, 1, 64, 256)
    m6 = _mat(lw.LW_FMT_Q6, 2, 64, 256)
    d4, d6 = _upload(lw.LW_FMT_Q4_PAIR, m4), _upload(lw.LW_FMT_Q6, m6)
    x = torch.zeros(256, device=DEV)
    y = torch.zeros(64, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    ws = torch.zeros(1 << 20, device=DEV)
    with pytest.raises(lw.LwError):
        lw.lw_decode_gemv_group([d4, d6], [x, x], [y, y], ws, st)          # mixed formats
    with pytest.raises(lw.LwError):
        lw.lw_decode_gemv_group([d4] * 9, [x] * 9, [y] * 9, ws, st)         # too many
    with pytest.raises(lw.LwError):
        lw.lw_decode_gemv_group([d4, d4], [x, x], [y, y], ws[:4], st)      # workspace too small
    hb = lw.lw_encode_bundle(lw.LW_FMT_Q4_PAIR, m4["codes"], m4["scales"], m4["mins"], twin=True)
    with pytest.raises(lw.LwError):
        lw.lw_decode_gemv_group([lw.DeviceBundle.upload(hb, DEV)], [x], [y], ws, st)   # twin
    assert int(st.item()) == 0


@pytest.mark.parametrize("fmt", [lw.LW_FMT_Q4_PAIR, lw.LW_FMT_Q6])
def test_twin_group_equals_single_twin_calls(fmt):
    n = 5
    mats = [_mat(fmt, 300 + i, *SHAPES[i]) for i in range(n)]
    tws = [lw.DeviceBundle.upload(lw.lw_encode_bundle(fmt, m["codes"], m["scales"], m.get("mins"),
                                                      twin=True), DEV) for m in mats]
    dbs = [_upload(fmt, m) for m in mats]
    xs = [torch.from_numpy(m["x"][0]).to(DEV) for m in mats]
    ys = [torch.full((d.rows,), float("nan"), device=DEV) for d in tws]
    ws = torch.zeros(lw.lw_workspace_bytes_group(tws) // 4 + 64, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    lw.lw_twin_gemv_group(tws, xs, ys, ws, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for d, t, x, y in zip(dbs, tws, xs, ys):
        y1 = torch.empty(t.rows, device=DEV)
        w1 = torch.zeros(lw.lw_workspace_bytes(t, 1) // 4 + 64, device=DEV)
        lw.lw_twin_gemv(t, x, y1, w1, st)
        torch.cuda.synchronize()
        yg = y.cpu().numpy()
        assert np.array_equal(yg.view(np.uint32), y1.cpu().numpy().view(np.uint32))
        # the twin executes the coded kernel's floating-point operations
        assert np.array_equal(yg.view(np.uint32), _single(d, x).view(np.uint32))
    with pytest.raises(lw.LwError):
        lw.lw_twin_gemv_group(dbs[:2], xs[:2], ys[:2], ws, st)        # coded bundles
    with pytest.raises(lw.LwError):
        lw.lw_twin_gemv_group([tws[0], dbs[1]], xs[:2], ys[:2], ws, st)   # mixed
    assert int(st.item()) == 0


def test_prepared_calls_equal_direct_calls():
    """PreparedGemv (arguments marshalled once) gives what the direct calls
    give, for one matrix, a group, and the twins."""
    fmt = lw.LW_FMT_Q4_PAIR
    mats = [_mat(fmt, 500 + i, *SHAPES[i]) for i in range(3)]
    dbs = [_upload(fmt, m) for m in mats]
    tws = [lw.DeviceBundle.upload(lw.lw_encode_bundle(fmt, m["codes"], m["scales"], m["mins"],
                                                      twin=True), DEV) for m in mats]
    xs = [torch.from_numpy(m["x"][0]).to(DEV) for m in mats]
    ws = torch.zeros(lw.lw_workspace_bytes_group(dbs) // 4 + 64, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    for bundles, twin in ((dbs, False), (tws, True)):
        for sel in ([0], [0, 1, 2]):
            ys = [torch.full((bundles[j].rows,), float("nan"), device=DEV) for j in sel]
            call = lw.PreparedGemv([bundles[j] for j in sel], [xs[j] for j in sel], ys, ws, st, twin=twin)
            call()
            call()
            torch.cuda.synchronize()
            assert int(st.item()) == 0
            for j, y in zip(sel, ys):
                ref = _single(dbs[j], xs[j])    # the twin gives the coded result bitwise
                assert np.array_equal(y.cpu().numpy().view(np.uint32), ref.view(np.uint32))


def test_step_graph_replays_the_calls():
    """lw_graph_begin / lw_graph_end / lw_graph_launch: a step of library
    calls (a group and a single matrix) captured once and replayed gives the
    eager results bitwise; capture refuses the default stream."""
    fmt = lw.LW_FMT_Q4_PAIR
    mats = [_mat(fmt, 700 + i, *SHAPES[i]) for i in range(3)]
    dbs = [_upload(fmt, m) for m in mats]
    xs = [torch.from_numpy(m["x"][0]).to(DEV) for m in mats]
    ys = [torch.full((d.rows,), float("nan"), device=DEV) for d in dbs]
    ws = torch.zeros(lw.lw_workspace_bytes_group(dbs[:2]) // 4 + 64, device=DEV)
    ws2 = torch.zeros(lw.lw_workspace_bytes(dbs[2], 1) // 4 + 64, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    calls = [lw.PreparedGemv(dbs[:2], xs[:2], ys[:2], ws, st), lw.PreparedGemv(dbs[2:], xs[2:], ys[2:], ws2, st)]
    for c in calls:
        c()                                   # eager once (launch attributes set up)
    torch.cuda.synchronize()
    ref = [y.cpu().numpy().copy() for y in ys]
    for y in ys:
        y.fill_(float("nan"))
    s = torch.cuda.Stream()
    g = lw.StepGraph(s)
    with g.capture():
        for c in calls:
            c()
    torch.cuda.synchronize()
    assert all(torch.isnan(y).all() for y in ys)      # captured, not run
    for _ in range(3):
        g.launch()
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for y, r in zip(ys, ref):
        assert np.array_equal(y.cpu().numpy().view(np.uint32), r.view(np.uint32))
    with pytest.raises(lw.LwError):
        lw._check(lw.load().lw_graph_begin(None), "lw_graph_begin")


@pytest.mark.parametrize("fmt", [lw.LW_FMT_Q4_PAIR, lw.LW_FMT_Q6])
@pytest.mark.parametrize("batch", [2, 3, 8])
def test_gemm_group_equals_per_matrix_products(fmt, batch):
    """lw_decode_gemm_group / lw_twin_gemm_group: batches of up to 8 rows in
    one launch, each output bitwise what the per-matrix CUDA-core product
    gives (these matrices stay on the CUDA cores up to 8 rows)."""
    n = 4
    mats = [(inputs.small_q4(900 + i, *SHAPES[i], batch=batch) if fmt == lw.LW_FMT_Q4_PAIR
             else inputs.small_q6(900 + i, *SHAPES[i], batch=batch)) for i in range(n)]
    dbs = [_upload(fmt, m) for m in mats]
    tws = [lw.DeviceBundle.upload(lw.lw_encode_bundle(fmt, m["codes"], m["scales"], m.get("mins"),
                                                      twin=True), DEV) for m in mats]
    Xs = [torch.from_numpy(np.ascontiguousarray(m["x"][:batch])).to(DEV) for m in mats]
    ws = torch.zeros(lw.lw_workspace_bytes_group(dbs) // 4 + 64, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    for bundles, group, one in ((dbs, lw.lw_decode_gemm_group, lw.lw_decode_gemm),
                                (tws, lw.lw_twin_gemm_group, lw.lw_twin_gemm)):
        Ys = [torch.full((batch, d.rows), float("nan"), device=DEV) for d in bundles]
        group(bundles, Xs, batch, Ys, ws, st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        for d, X, Y in zip(bundles, Xs, Ys):
            Y1 = torch.empty(batch, d.rows, device=DEV)
            w1 = torch.zeros(lw.lw_workspace_bytes(d, batch) // 4 + 64, device=DEV)
            one(d, X, batch, Y1, w1, st)
            torch.cuda.synchronize()
            assert np.array_equal(Y.cpu().numpy().view(np.uint32), Y1.cpu().numpy().view(np.uint32))
    for m, Y in zip(mats, Ys):
        ref = oracle.reference_output(oracle.Q4 if fmt == lw.LW_FMT_Q4_PAIR else oracle.Q6, m)
        scale = oracle.abs_row_products(oracle.Q4 if fmt == lw.LW_FMT_Q4_PAIR else oracle.Q6, m)
        assert_close(Y.cpu().numpy(), ref, scale)
    with pytest.raises(lw.LwError):
        lw.lw_decode_gemm_group(dbs, Xs, 9, Ys, ws, st)
    assert int(st.item()) == 0
