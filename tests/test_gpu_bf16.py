"""GPU parity of the BF16 exponent-coded path through the C ABI against the
CPU oracle: decode bit-exact (coded and direct-palette twin), products within
tolerance, twin bitwise equal to the coded kernel, verbatim-heavy and
verbatim-free matrices, batches, and the Llama-3.1-8B MLP at full size on
sampled outputs."""
import numpy as np
import pytest

import oracle
from decode_gemv_gb300 import inputs
from decode_gemv_gb300 import lw
from helpers import assert_close

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
DEV = "cuda"
FMT = lw.LW_FMT_BF16_EXP


@pytest.fixture(scope="module", autouse=True)
def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lw.load()


def upload(bits, twin=False):
    hb = lw.lw_encode_bundle(FMT, bits, twin=twin)
    return hb, lw.DeviceBundle.upload(hb, DEV)


def run_decode(db):
    out = torch.zeros(db.rows * db.cols, dtype=torch.int16, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    lw.lw_decode(db, out, st)
    torch.cuda.synchronize()
    return out.cpu().numpy().view(np.uint16).reshape(db.rows, db.cols), int(st.item())


def run_product(db, xbits, twin=False):
    B = xbits.shape[0]
    X = torch.from_numpy(np.ascontiguousarray(xbits).view(np.int16)).to(DEV)
    Y = torch.full((B, db.rows), float("nan"), dtype=torch.float32, device=DEV)
    ws = torch.zeros(max(1, lw.lw_workspace_bytes(db, B) // 4), dtype=torch.float32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    if twin:
        lw.lw_twin_gemm(db, X, B, Y, ws, st)
    else:
        lw.lw_decode_gemm(db, X, B, Y, ws, st)
    torch.cuda.synchronize()
    return Y.cpu().numpy(), int(st.item())


def all_verbatim(bits):
    r, k = np.indices(bits.shape)
    exp = (100 + (r * 7 + k) % 16).astype(np.uint16)
    exp[:, ::64] = 200 + (r[:, ::64] * 8 + k[:, ::64] // 64) % 40
    return ((bits & 0x807F) | (exp << 7)).astype(np.uint16)


CASES = [((64, 256), 0.002), ((192, 768), 0.002), ((128, 1024), 0.02), ((256, 512), 0.0),
         ((128, 3072), 0.002)]


@pytest.mark.parametrize("shape,p", CASES)
def test_bf16_decode_bit_exact(shape, p):
    n, k = shape
    m = inputs.small_bf16(n + k, n, k, outlier_p=p)
    for twin in (False, True):
        _, db = upload(m["bits"], twin)
        out, st = run_decode(db)
        assert st == 0
        assert np.array_equal(out, m["bits"])


def test_bf16_decode_all_verbatim():
    m = inputs.small_bf16(3, 128, 512)
    bits = all_verbatim(m["bits"])
    hb, db = upload(bits)
    assert hb.stats.n_verbatim == 128 * 8
    out, st = run_decode(db)
    assert st == 0 and np.array_equal(out, bits)
    x = m["x"]
    y, st = run_product(db, x)
    assert st == 0
    mm = dict(bits=bits, x=x)
    assert_close(y, oracle.reference_output(oracle.BF16, mm), oracle.abs_row_products(oracle.BF16, mm))


@pytest.mark.parametrize("shape,p", CASES)
def test_bf16_gemv_parity_and_twin_bitwise(shape, p):
    n, k = shape
    m = inputs.small_bf16(3 * n + k, n, k, outlier_p=p)
    _, db = upload(m["bits"])
    _, dt = upload(m["bits"], twin=True)
    y, st = run_product(db, m["x"])
    assert st == 0
    yt, st = run_product(dt, m["x"], twin=True)
    assert st == 0
    assert_close(y, oracle.reference_output(oracle.BF16, m), oracle.abs_row_products(oracle.BF16, m))
    assert np.array_equal(y.view(np.uint32), yt.view(np.uint32))


@pytest.mark.parametrize("batch", [2, 4, 5, 8, 12])
def test_bf16_gemm_batches(batch):
    m = inputs.small_bf16(40 + batch, 192, 1024, batch=batch)
    _, db = upload(m["bits"])
    Y, st = run_product(db, m["x"])
    assert st == 0
    assert_close(Y, oracle.reference_output(oracle.BF16, m), oracle.abs_row_products(oracle.BF16, m))
    y1, _ = run_product(db, m["x"][:1])
    assert np.array_equal(Y[0].view(np.uint32), y1[0].view(np.uint32))


def test_bf16_corrupt_word_reported():
    m = inputs.small_bf16(9, 128, 512)
    hb = lw.lw_encode_bundle(FMT, m["bits"])
    words = hb.view("words", np.uint32).copy()
    toff = hb.view("tile_off", np.uint32)
    words[toff[2] * 32 + 5] ^= np.uint32(0xF0000000)
    secs = dict(hb.sections, words=words.view(np.uint8))
    db = lw.DeviceBundle(FMT, False, 128, 512, secs, hb.stats.max_tile_rows, hb.stats.min_len,
                         hb.stats.max_len, DEV)
    _, st = run_decode(db)
    _, st2 = run_product(db, m["x"])
    # a flipped word almost always changes where the lane's codes end; either
    # way nothing faults and the status is one of the documented codes
    assert st in (0, 1) and st2 in (0, 1)


@pytest.mark.parametrize("index", range(3))
def test_full_size_llama_mlp(index):
    spec = inputs.workload_specs(inputs.LLAMA_MLP_BF16)[index]
    m = inputs.make_matrix(inputs.LLAMA_MLP_BF16, spec, 0, index, batch=4)
    _, db = upload(m["bits"])
    out, st = run_decode(db)
    assert st == 0 and np.array_equal(out, m["bits"])
    rows = np.unique(np.concatenate([np.arange(0, spec.rows, max(1, spec.rows // 64)), [spec.rows - 1]]))
    sub = dict(bits=m["bits"][rows], x=m["x"])
    ref = oracle.reference_output(oracle.BF16, sub)
    absprod = oracle.abs_row_products(oracle.BF16, sub)
    for b in (1, 4):
        Y, st = run_product(db, m["x"][:b])
        assert st == 0
        assert_close(Y[:, rows], ref[:b], absprod[:b])
    del db
    _, dt = upload(m["bits"], twin=True)
    Yt, st = run_product(dt, m["x"][:1], twin=True)
    assert st == 0
    Y1, _ = run_product(upload(m["bits"])[1], m["x"][:1])
    assert np.array_equal(Y1.view(np.uint32), Yt.view(np.uint32))


@pytest.mark.parametrize("shape,batch", [((256, 1024), 16), ((192, 768), 17), ((512, 512), 32),
                                         ((256, 2048), 48), ((320, 1024), 64), ((128, 256), 64),
                                         ((256, 1024), 80)])
def test_bf16_tensor_core_batches(shape, batch):
    """Batches >= 16 take the tcgen05 path (BF16 rebuilt in shared memory,
    FP32 accumulation in tensor memory); checked against the oracle and
    against the CUDA-core path fed 8 activation rows at a time."""
    n, k = shape
    m = inputs.small_bf16(5 * n + batch, n, k, batch=batch)
    _, db = upload(m["bits"])
    Y, st = run_product(db, m["x"])
    assert st == 0
    ref = oracle.reference_output(oracle.BF16, m)
    absprod = oracle.abs_row_products(oracle.BF16, m)
    assert_close(Y, ref, absprod)
    Yc = np.concatenate([run_product(db, m["x"][b: b + 8])[0] for b in range(0, batch, 8)])
    assert_close(Y, Yc, absprod)
    Y2, st = run_product(db, m["x"])           # twice in a row: counters reset
    assert st == 0 and np.array_equal(Y.view(np.uint32), Y2.view(np.uint32))
    # the direct-palette twin on the tensor cores: the same operands, so
    # bitwise the coded product
    _, dt = upload(m["bits"], twin=True)
    Yt, st = run_product(dt, m["x"], twin=True)
    assert st == 0 and np.array_equal(Y.view(np.uint32), Yt.view(np.uint32))


def test_bf16_twin_tensor_core_all_verbatim_and_none():
    """Direct-palette twin on the tensor cores with every 64-group verbatim,
    and with none: against the oracle and bitwise against the coded product."""
    for kind in ("all", "none"):
        m = inputs.small_bf16(77, 256, 1024, batch=32, outlier_p=0.0)
        if kind == "all":
            m["bits"] = all_verbatim(m["bits"])
        _, db = upload(m["bits"])
        _, dt = upload(m["bits"], twin=True)
        Y, st = run_product(db, m["x"])
        Yt, stt = run_product(dt, m["x"], twin=True)
        assert st == 0 and stt == 0
        assert_close(Yt, oracle.reference_output(oracle.BF16, m), oracle.abs_row_products(oracle.BF16, m))
        assert np.array_equal(Y.view(np.uint32), Yt.view(np.uint32))


def test_bf16_tensor_core_full_size_down():
    spec = inputs.workload_specs(inputs.LLAMA_MLP_BF16)[2]
    m = inputs.make_matrix(inputs.LLAMA_MLP_BF16, spec, 0, 2, batch=64)
    _, db = upload(m["bits"])
    rows = np.unique(np.concatenate([np.arange(0, spec.rows, 97), [spec.rows - 1]]))
    sub = dict(bits=m["bits"][rows], x=m["x"])
    for b in (16, 64):
        Y, st = run_product(db, m["x"][:b])
        assert st == 0
        assert_close(Y[:, rows], oracle.reference_output(oracle.BF16, dict(sub, x=m["x"][:b])),
                     oracle.abs_row_products(oracle.BF16, dict(sub, x=m["x"][:b])))
