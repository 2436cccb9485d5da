"""lw_decode_gemv_noalloc: the allocation-free variant of the fused decode +
GEMV (scratch in a fixed device array inside the library) for callers that
cannot allocate device memory -- e.g. code under CUDA-graph capture or an
engine whose own pool owns all device memory.  Checked through the C ABI
against lw_decode_gemv with a caller workspace, on two calls in a row, for
the 4-bit, 6-bit and BF16-exponent formats (the argument checks that run
before the shared counters are cleared are covered on the CPU).  This
file is collected last so that a run stopping at the first failure has run
everything else; it also passes alone in a fresh process (the first call then
sets the scratch up)."""
import numpy as np
import pytest

from decode_gemv_gb300 import inputs
from decode_gemv_gb300 import lw
from helpers import TOL, rel_errors

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lw.load()


def _bundle(m, fmt):
    payload = m["bits"] if fmt == lw.LW_FMT_BF16_EXP else m["codes"]
    hb = lw.lw_encode_bundle(fmt, payload, m.get("scales"), m.get("mins"))
    return lw.DeviceBundle.upload(hb, "cuda")


def _with_workspace(db, x):
    y = torch.empty(db.rows, dtype=torch.float32, device="cuda")
    ws = torch.zeros(lw.lw_workspace_bytes(db, 1) // 4, dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    lw.lw_decode_gemv(db, x, y, ws, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return y.cpu().numpy()


def _no_alloc(db, x):
    y = torch.full((db.rows,), float("nan"), dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    lw.lw_decode_gemv_noalloc(db, x, y, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return y.cpu().numpy()


@pytest.mark.parametrize("fmt,shape", [(lw.LW_FMT_Q4_PAIR, (256, 1024)),
                                       (lw.LW_FMT_Q6, (192, 768)),
                                       (lw.LW_FMT_Q4_PAIR, (4096, 14336)),
                                       (lw.LW_FMT_BF16_EXP, (256, 1024))])
def test_no_alloc_matches_workspace_entry_point(fmt, shape):
    n, k = shape
    make = {lw.LW_FMT_Q4_PAIR: inputs.small_q4, lw.LW_FMT_Q6: inputs.small_q6,
            lw.LW_FMT_BF16_EXP: inputs.small_bf16}[fmt]
    m = make(101, n, k, batch=2)
    db = _bundle(m, fmt)
    assert lw.lw_workspace_bytes(db, 1) <= lw.lw_noalloc_scratch_bytes()
    # two calls in a row, with different activations: the second must not see
    # anything the first left in the shared scratch
    for b in (0, 1):
        xb = np.ascontiguousarray(m["x"][b])
        if fmt == lw.LW_FMT_BF16_EXP:
            xb = xb.view(np.int16)    # bf16 bits
        x = torch.from_numpy(xb).to("cuda")
        want = _with_workspace(db, x)
        got = _no_alloc(db, x)
        nw = rel_errors(got, want, np.abs(want) + 1e-30)[0]
        assert nw <= TOL
        assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


def test_no_alloc_rejects_matrices_beyond_its_scratch():
    m = inputs.small_q4(5, 64, 256)
    db = _bundle(m, lw.LW_FMT_Q4_PAIR)
    db.view.rows = 64 * 1024          # claims a matrix far larger than the scratch
    db.view.cols = 256 * 64
    x = torch.zeros(db.view.cols, dtype=torch.float32, device="cuda")   # sized for the claim,
    y = torch.zeros(db.view.rows, dtype=torch.float32, device="cuda")   # so only the scratch limit refuses
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(lw.LwError) as e:
        lw.lw_decode_gemv_noalloc(db, x, y, st)
    assert e.value.status == 3 and "scratch" in str(e.value)
