"""Tile-skip launch lists (lw_decode_gemm_strips): the product over a list of
64-row strips ("Software-Defined Bandwidth Expansion" §IV.C, an inactive tile
absent from a smaller launch grid).  Listed rows are bitwise what the full
product gives (and within tolerance of the oracle); every other row is left
untouched; bad list entries are reported and skipped; host errors."""
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


def _setup(fmt, n, k, batch, seed):
    m = (inputs.small_q4(seed, n, k, batch=batch) if fmt == lw.LW_FMT_Q4_PAIR
         else inputs.small_q6(seed, n, k, batch=batch))
    hb = lw.lw_encode_bundle(fmt, m["codes"], m["scales"], m.get("mins"))
    db = lw.DeviceBundle.upload(hb, DEV)
    X = torch.from_numpy(np.ascontiguousarray(m["x"][:batch])).to(DEV)
    ws = torch.zeros(lw.lw_workspace_bytes(db, batch) // 4 + 64, device=DEV)
    return m, db, X, ws


def _full(db, X, batch, ws):
    """The full product in slices of up to 8 rows (CUDA-core passes: the
    strip-list product sums in their order)."""
    Y = torch.empty(batch, db.rows, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    for b0 in range(0, batch, 8):
        nb = min(8, batch - b0)
        lw.lw_decode_gemm(db, X[b0:b0 + nb].contiguous(), nb, Y[b0:b0 + nb], ws, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return Y.cpu().numpy()


def _strips(db, X, batch, ws, lst):
    Y = torch.full((batch, db.rows), float("nan"), device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    s = torch.tensor(lst, dtype=torch.int32, device=DEV)
    lw.lw_decode_gemm_strips(db, s, X, batch, Y, ws, st)
    torch.cuda.synchronize()
    return Y.cpu().numpy(), int(st.item())


def _rows(lst):
    return np.concatenate([np.arange(64 * s, 64 * s + 64) for s in lst]) if len(lst) else np.zeros(0, int)


@pytest.mark.parametrize("fmt", [lw.LW_FMT_Q4_PAIR, lw.LW_FMT_Q6])
@pytest.mark.parametrize("batch", [1, 3, 11])
def test_listed_rows_match_the_full_product(fmt, batch):
    n, k = 640, 1024
    m, db, X, ws = _setup(fmt, n, k, batch, 40 + batch)
    full = _full(db, X, batch, ws)
    rng = np.random.default_rng(batch)
    for lst in ([], [0], [9], [1, 4, 5, 8], list(range(10)), sorted(rng.choice(10, 6, replace=False).tolist())):
        y, st = _strips(db, X, batch, ws, lst)
        assert st == 0
        r = _rows(lst)
        assert np.array_equal(y[:, r].view(np.uint32), full[:, r].view(np.uint32))
        other = np.setdiff1d(np.arange(n), r)
        assert np.isnan(y[:, other]).all()
    # the listed rows against the oracle
    lst = [2, 3, 7]
    y, st = _strips(db, X, batch, ws, lst)
    r = _rows(lst)
    ref = oracle.reference_output(oracle.Q4 if fmt == lw.LW_FMT_Q4_PAIR else oracle.Q6, m)
    scale = oracle.abs_row_products(oracle.Q4 if fmt == lw.LW_FMT_Q4_PAIR else oracle.Q6, m)
    assert_close(y[:, r], ref[:, r], scale[:, r])


def test_bad_entries_are_reported_and_skipped():
    n, k = 512, 512
    m, db, X, ws = _setup(lw.LW_FMT_Q4_PAIR, n, k, 1, 7)
    full = _full(db, X, 1, ws)
    for lst, good in (([1, 3, 99], [1, 3]), ([2, 2, 5], [2, 5]), ([4, 1, 6], [4, 6]), ([-1, 0, 7], [0, 7])):
        y, st = _strips(db, X, 1, ws, lst)
        assert st == 6                      # LW_DEV_BAD_STRIPS
        r = _rows(good)
        assert np.array_equal(y[:, r].view(np.uint32), full[:, r].view(np.uint32))
    # the workspace counters are left at zero: a clean call afterwards
    y, st = _strips(db, X, 1, ws, [0, 1, 2, 3, 4, 5, 6, 7])
    assert st == 0 and np.array_equal(y.view(np.uint32), full.view(np.uint32))


def test_host_errors():
    m, db, X, ws = _setup(lw.LW_FMT_Q4_PAIR, 128, 256, 1, 8)
    Y = torch.empty(1, 128, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    s = torch.tensor([0, 1, 2], dtype=torch.int32, device=DEV)
    with pytest.raises(lw.LwError):
        lw.lw_decode_gemm_strips(db, s, X, 1, Y, ws, st)         # 3 entries > 2 strips
    with pytest.raises(lw.LwError):
        lw.lw_decode_gemm_strips(db, s[:1], X, 1, Y, ws[:1], st)  # workspace too small
    mb = inputs.small_bf16(9, 64, 256)
    dbb = lw.DeviceBundle.upload(lw.lw_encode_bundle(lw.LW_FMT_BF16_EXP, mb["bits"]), DEV)
    with pytest.raises(lw.LwError) as e:
        lw.lw_decode_gemm_strips(dbb, s[:1], X.to(torch.bfloat16), 1, Y[:, :64], ws, st)
    assert e.value.status == lw.LW_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert int(st.item()) == 0
