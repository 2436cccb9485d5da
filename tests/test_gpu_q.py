"""GPU parity of the 4-/6-bit paths through the C ABI against the CPU oracle:
decode bit-exact, products within tolerance, twin bitwise equal to the coded
kernel, batches, cross-decoding of oracle-built bundles, corruption reports,
edge cases, and the full-size workloads on sampled outputs."""
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


def upload(fmt, m, twin=False):
    hb = lw.lw_encode_bundle(fmt, m["codes"], m["scales"], m.get("mins"), twin=twin)
    return hb, lw.DeviceBundle.upload(hb, DEV)


def status():
    return torch.zeros(1, dtype=torch.int32, device=DEV)


def run_product(db, x, twin=False, stream=None):
    """x: numpy [B][K] fp32.  Returns Y numpy [B][N] and the device status."""
    B = x.shape[0]
    X = torch.from_numpy(np.ascontiguousarray(x)).to(DEV)
    Y = torch.full((B, db.rows), float("nan"), dtype=torch.float32, device=DEV)
    ws = torch.zeros(max(1, lw.lw_workspace_bytes(db, B) // 4), dtype=torch.float32, device=DEV)
    st = status()
    if twin:
        (lw.lw_twin_gemv if B == 1 else lambda *a, **k: lw.lw_twin_gemm(a[0], a[1], B, *a[2:], **k))(
            db, X, Y, ws, st, stream=stream)
    elif B == 1:
        lw.lw_decode_gemv(db, X, Y, ws, st, stream=stream)
    else:
        lw.lw_decode_gemm(db, X, B, Y, ws, st, stream=stream)
    torch.cuda.synchronize()
    return Y.cpu().numpy(), int(st.item())


def run_decode(db):
    fmt = db.fmt
    nbytes = db.rows * db.cols // 2 if fmt == lw.LW_FMT_Q4_PAIR else db.rows * db.cols
    out = torch.zeros(nbytes, dtype=torch.uint8, device=DEV)
    st = status()
    lw.lw_decode(db, out, st)
    torch.cuda.synchronize()
    shape = (db.rows, db.cols // 2) if fmt == lw.LW_FMT_Q4_PAIR else (db.rows, db.cols)
    return out.cpu().numpy().reshape(shape), int(st.item())


def expect_codes(fmt, codes):
    return oracle.q4_pair_symbols(codes).astype(np.uint8) if fmt == lw.LW_FMT_Q4_PAIR else codes


SHAPES = [(64, 256), (192, 768), (256, 1024), (128, 3072), (320, 512)]


@pytest.mark.parametrize("twin", [False, True])
@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("fmt", [lw.LW_FMT_Q4_PAIR, lw.LW_FMT_Q6])
def test_decode_bit_exact(fmt, shape, twin):
    n, k = shape
    m = inputs.small_q4(n + k, n, k, sd=1.2 + (n % 3) * 0.5) if fmt == lw.LW_FMT_Q4_PAIR \
        else inputs.small_q6(n + k, n, k)
    _, db = upload(fmt, m, twin)
    out, st = run_decode(db)
    assert st == 0
    assert np.array_equal(out, expect_codes(fmt, m["codes"]))


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("fmt", [lw.LW_FMT_Q4_PAIR, lw.LW_FMT_Q6])
def test_gemv_parity_and_twin_bitwise(fmt, shape):
    n, k = shape
    m = inputs.small_q4(7 * n + k, n, k, sd=1.6) if fmt == lw.LW_FMT_Q4_PAIR \
        else inputs.small_q6(7 * n + k, n, k)
    _, db = upload(fmt, m)
    _, dt = upload(fmt, m, twin=True)
    y, st = run_product(db, m["x"])
    assert st == 0
    yt, stt = run_product(dt, m["x"], twin=True)
    assert stt == 0
    ref = oracle.reference_output(fmt, m)
    assert_close(y, ref, oracle.abs_row_products(fmt, m))
    assert np.array_equal(y.view(np.uint32), yt.view(np.uint32)), "twin and coded kernel differ"


@pytest.mark.parametrize("batch", [1, 2, 3, 4, 5])
@pytest.mark.parametrize("fmt", [lw.LW_FMT_Q4_PAIR, lw.LW_FMT_Q6])
def test_gemm_batches(fmt, batch):
    n, k = 192, 1024
    m = inputs.small_q4(31 + batch, n, k, batch=batch) if fmt == lw.LW_FMT_Q4_PAIR \
        else inputs.small_q6(31 + batch, n, k, batch=batch)
    _, db = upload(fmt, m)
    Y, st = run_product(db, m["x"])
    assert st == 0
    ref = oracle.reference_output(fmt, m)
    assert_close(Y, ref, oracle.abs_row_products(fmt, m))
    # every activation row gives bitwise what a batch-1 call gives
    for b in (0, batch - 1):
        y1, _ = run_product(db, m["x"][b: b + 1])
        assert np.array_equal(Y[b].view(np.uint32), y1[0].view(np.uint32))
    _, dt = upload(fmt, m, twin=True)
    Yt, stt = run_product(dt, m["x"], twin=True)
    assert stt == 0 and np.array_equal(Y.view(np.uint32), Yt.view(np.uint32))


# tensor-core passes: from 6 rows for matrices with at least 1.5 (256-row
# block x K split) units per SM, from 9 rows for any matrix
TC_CASES = [((2048, 16384), 6), ((8192, 4096), 12), ((4096, 8192), 16), ((2048, 16384), 33),
            ((4096, 8192), 40), ((192, 1024), 7), ((192, 1024), 12), ((64, 256), 32),
            ((320, 512), 70)]


@pytest.mark.parametrize("shape,batch", TC_CASES)
@pytest.mark.parametrize("fmt", [lw.LW_FMT_Q4_PAIR, lw.LW_FMT_Q6])
def test_tensor_core_batches(fmt, shape, batch):
    """Batches of 6 or more rows take the tcgen05 path (weights and
    activations split into BF16 high and low parts, FP32 accumulation in
    tensor memory): against the oracle, against the CUDA-core path fed 4
    rows at a time, against the twin, and deterministic."""
    n, k = shape
    m = inputs.small_q4(3 * n + batch, n, k, batch=batch) if fmt == lw.LW_FMT_Q4_PAIR \
        else inputs.small_q6(3 * n + batch, n, k, batch=batch)
    _, db = upload(fmt, m)
    Y, st = run_product(db, m["x"])
    assert st == 0
    absprod = oracle.abs_row_products(fmt, m)
    assert_close(Y, oracle.reference_output(fmt, m), absprod)
    Yc = np.concatenate([run_product(db, m["x"][b: b + 4])[0] for b in range(0, batch, 4)])
    assert_close(Y, Yc, absprod)
    _, dt = upload(fmt, m, twin=True)
    Yt, stt = run_product(dt, m["x"], twin=True)
    assert stt == 0
    assert_close(Y, Yt, absprod)
    Y2, st2 = run_product(db, m["x"])
    assert st2 == 0 and np.array_equal(Y.view(np.uint32), Y2.view(np.uint32))


def test_oracle_built_bundle_decodes_on_gpu():
    """Cross-decoding: sections written by the oracle's encoder, table rebuilt
    from its code lengths, decoded and multiplied by the CUDA path."""
    n, k = 192, 1024
    m = inputs.small_q4(77, n, k, sd=1.9)
    ob = oracle.encode(oracle.Q4, m["codes"])
    hb = lw.lw_encode_bundle(lw.LW_FMT_Q4_PAIR, m["codes"], m["scales"], m["mins"])
    table = lw.lw_table_from_lengths(lw.LW_FMT_Q4_PAIR, ob["code_len"])
    tf = lw.table_fields(table)
    secs = dict(words=ob["words"], tile_off=ob["tile_off"], lane_bits=ob["lane_bits"],
                table=table, qparams=hb.sections["qparams"], lane_mid=ob["lane_mid"])
    wt = int(np.diff(ob["tile_off"]).max())
    lw.lw_validate_sections(lw.LW_FMT_Q4_PAIR, n, k, secs, wt)
    db = lw.DeviceBundle(lw.LW_FMT_Q4_PAIR, False, n, k, secs, wt, tf["lmin"], tf["lmax"], DEV)
    out, st = run_decode(db)
    assert st == 0 and np.array_equal(out, expect_codes(lw.LW_FMT_Q4_PAIR, m["codes"]))
    y, st = run_product(db, m["x"])
    assert st == 0
    assert_close(y, oracle.reference_output(oracle.Q4, m), oracle.abs_row_products(oracle.Q4, m))


def test_corrupted_words_are_reported_not_trapped():
    n, k = 128, 512
    m = inputs.small_q4(5, n, k)
    hb = lw.lw_encode_bundle(lw.LW_FMT_Q4_PAIR, m["codes"], m["scales"], m["mins"])
    words = hb.view("words", np.uint32).copy()
    toff = hb.view("tile_off", np.uint32)
    # flip one bit of lane 3 of tile 1, choosing the first bit whose flip the
    # oracle sees as a lane that no longer ends at its recorded length
    tf = lw.table_fields(hb.sections["table"])
    nsym = np.full((len(toff) - 1, 32), 256, np.int32)
    want = hb.view("lane_bits", np.uint16).reshape(-1, 32)[1, 3]
    for bit in range(31, -1, -1):
        trial = words.copy()
        trial[toff[1] * 32 + 3] ^= np.uint32(1 << bit)
        _, used = oracle.decode_lanes(tf["code_len"], trial, toff, nsym, 256)
        if used[1, 3] != want:
            words = trial
            break
    else:
        pytest.fail("no detectable single-bit flip in the first word")
    secs = dict(hb.sections, words=words.view(np.uint8))
    db = lw.DeviceBundle(lw.LW_FMT_Q4_PAIR, False, n, k, secs, hb.stats.max_tile_rows,
                         hb.stats.min_len, hb.stats.max_len, DEV)
    _, st = run_decode(db)
    assert st == 1
    _, st = run_product(db, m["x"])
    assert st == 1


def test_bad_device_table_is_rejected_in_kernel():
    m = inputs.small_q4(6, 64, 256)
    hb, db = upload(lw.LW_FMT_Q4_PAIR, m)
    t = db.tensors["table"]
    off0 = t[80:84].view(torch.int32)
    off0 += 100000          # would index far outside the symbol table
    y, st = run_product(db, m["x"])
    assert st == 5
    _, st = run_decode(db)
    assert st == 5


def test_host_argument_errors():
    m = inputs.small_q4(8, 64, 256)
    hb, db = upload(lw.LW_FMT_Q4_PAIR, m)
    x = torch.zeros(256, dtype=torch.float32, device=DEV)
    y = torch.zeros(64, dtype=torch.float32, device=DEV)
    ws = torch.zeros(1, dtype=torch.float32, device=DEV)   # too small
    with pytest.raises(lw.LwError) as e:
        lw.lw_decode_gemv(db, x, y, ws, status())
    assert e.value.status == 1
    db.view.rows = 65
    ws = torch.zeros(1 << 16, dtype=torch.float32, device=DEV)
    with pytest.raises(lw.LwError) as e:
        lw.lw_decode_gemv(db, x, y, ws, status())
    assert e.value.status == 2
    db.view.rows = 64
    _, dt = upload(lw.LW_FMT_Q4_PAIR, m, twin=True)
    with pytest.raises(lw.LwError):
        lw.lw_decode_gemv(dt, x, y, ws, status())     # twin given to the coded call


def test_edge_single_symbol_and_long_lane():
    n, k = 64, 512
    m = inputs.small_q4(9, n, k)
    m["codes"] = np.full((n, k), 11, np.uint8)
    _, db = upload(lw.LW_FMT_Q4_PAIR, m)
    out, st = run_decode(db)
    assert st == 0 and np.array_equal(out, expect_codes(lw.LW_FMT_Q4_PAIR, m["codes"]))
    y, st = run_product(db, m["x"])
    assert st == 0
    assert_close(y, oracle.reference_output(oracle.Q4, m), oracle.abs_row_products(oracle.Q4, m))
    c = np.full((n, k), 7, np.uint8)
    c[:2, :256] = np.random.default_rng(0).integers(0, 16, size=(2, 256))
    m["codes"] = c
    hb, db = upload(lw.LW_FMT_Q4_PAIR, m)
    assert hb.stats.max_tile_rows > 20
    out, st = run_decode(db)
    assert st == 0 and np.array_equal(out, expect_codes(lw.LW_FMT_Q4_PAIR, c))
    y, st = run_product(db, m["x"])
    assert st == 0
    assert_close(y, oracle.reference_output(oracle.Q4, m), oracle.abs_row_products(oracle.Q4, m))


def test_runs_on_a_side_stream():
    m = inputs.small_q4(10, 256, 1024)
    _, db = upload(lw.LW_FMT_Q4_PAIR, m)
    s = torch.cuda.Stream()
    y, st = run_product(db, m["x"], stream=s)
    assert st == 0
    assert_close(y, oracle.reference_output(oracle.Q4, m), oracle.abs_row_products(oracle.Q4, m))


def sampled_reference(fmt, m, rows):
    """Oracle outputs for selected rows only (fp64, from the generator's codes)."""
    sub = dict(m)
    sub["codes"] = m["codes"][rows]
    sub["scales"] = m["scales"][rows]
    if m.get("mins") is not None:
        sub["mins"] = m["mins"][rows]
    return oracle.reference_output(fmt, sub), oracle.abs_row_products(fmt, sub)


@pytest.mark.parametrize("index", range(7))
def test_full_size_mistral_layer(index):
    """The Mistral-7B-shaped 4-bit layer at full size: decode bit-exact over the
    whole matrix, fused GEMV on sampled rows against the oracle, twin bitwise."""
    spec = inputs.workload_specs(inputs.MISTRAL_LAYER)[index]
    m = inputs.make_matrix(inputs.MISTRAL_LAYER, spec, 0, index)
    _, db = upload(spec.fmt, m)
    out, st = run_decode(db)
    assert st == 0 and np.array_equal(out, expect_codes(spec.fmt, m["codes"]))
    y, st = run_product(db, m["x"])
    assert st == 0
    rows = np.unique(np.concatenate([np.arange(0, spec.rows, max(1, spec.rows // 96)),
                                     [spec.rows - 1]]))
    ref, absprod = sampled_reference(spec.fmt, m, rows)
    assert_close(y[:, rows], ref, absprod)
    del db
    _, dt = upload(spec.fmt, m, twin=True)
    yt, st = run_product(dt, m["x"], twin=True)
    assert st == 0 and np.array_equal(y.view(np.uint32), yt.view(np.uint32))


@pytest.mark.parametrize("index", [4, 6])
def test_full_size_mistral_tensor_core(index):
    """gate (14336x4096) and down (4096x14336) at batch 16 and 32 on the
    tensor cores, sampled rows against the oracle."""
    spec = inputs.workload_specs(inputs.MISTRAL_LAYER)[index]
    m = inputs.make_matrix(inputs.MISTRAL_LAYER, spec, 0, index, batch=32)
    _, db = upload(spec.fmt, m)
    rows = np.unique(np.concatenate([np.arange(0, spec.rows, 131), [spec.rows - 1]]))
    ref, absprod = sampled_reference(spec.fmt, m, rows)
    for b in (16, 32):
        Y, st = run_product(db, m["x"][:b])
        assert st == 0
        assert_close(Y[:, rows], ref[:b], absprod[:b])


@pytest.mark.parametrize("index", range(4))
def test_full_size_phi3_layer(index):
    spec = inputs.workload_specs(inputs.PHI3_LAYER)[index]
    m = inputs.make_matrix(inputs.PHI3_LAYER, spec, 0, index, batch=8)
    _, db = upload(spec.fmt, m)
    out, st = run_decode(db)
    assert st == 0 and np.array_equal(out, m["codes"])
    rows = np.unique(np.concatenate([np.arange(0, spec.rows, max(1, spec.rows // 64)),
                                     [spec.rows - 1]]))
    ref, absprod = sampled_reference(spec.fmt, m, rows)
    for b in (1, 2, 4, 8):
        Y, st = run_product(db, m["x"][:b])
        assert st == 0
        assert_close(Y[:, rows], ref[:b], absprod[:b])
