"""Load-time transcode of a coded bundle into its fixed-width twin on the
device (lw_transcode_twin): the twin's words, tile offsets and lane bit
counts are bit-exact with the host twin builder and with the oracle's twin
layout; products on the transcoded twin equal the coded products bitwise;
corrupt streams are reported; bad views are refused on the host."""
import numpy as np
import pytest

import oracle
from decode_gemv_gb300 import inputs
from decode_gemv_gb300 import lw

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lw.load()


def _encode(fmt, m, twin=False):
    if fmt == lw.LW_FMT_BF16_EXP:
        return lw.lw_encode_bundle(fmt, m["bits"], twin=twin)
    return lw.lw_encode_bundle(fmt, m["codes"], m["scales"], m.get("mins"), twin=twin)


def _payload(fmt, m):
    return m["bits"] if fmt == lw.LW_FMT_BF16_EXP else m["codes"]


def _transcode(db):
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    tw = lw.lw_transcode_twin(db, st)
    torch.cuda.synchronize()
    return tw, int(st.item())


def _host(t, dtype):
    return t.cpu().numpy().view(dtype)


CASES = [
    (lw.LW_FMT_Q4_PAIR, lambda: inputs.small_q4(11, 192, 768)),
    (lw.LW_FMT_Q4_PAIR, lambda: inputs.small_q4(12, 64, 256, sd=0.3)),     # short codes
    (lw.LW_FMT_Q4_PAIR, lambda: inputs.small_q4(13, 128, 1024, sd=6.0)),   # long codes
    (lw.LW_FMT_Q6, lambda: inputs.small_q6(14, 128, 512)),
    (lw.LW_FMT_Q6, lambda: inputs.small_q6(15, 64, 2048)),
    (lw.LW_FMT_BF16_EXP, lambda: inputs.small_bf16(16, 128, 512)),
    (lw.LW_FMT_BF16_EXP, lambda: inputs.small_bf16(17, 64, 768, outlier_p=0.02)),   # many verbatim groups
    (lw.LW_FMT_BF16_EXP, lambda: inputs.small_bf16(18, 64, 256, outlier_p=0.0)),    # none
]


@pytest.mark.parametrize("fmt,make", CASES)
def test_transcoded_twin_is_bit_exact(fmt, make):
    m = make()
    hb, ht = _encode(fmt, m), _encode(fmt, m, twin=True)
    db = lw.DeviceBundle.upload(hb, DEV)
    tw, st = _transcode(db)
    assert st == 0
    words = _host(tw.tensors["words"], np.uint32)
    assert np.array_equal(words, ht.view("words", np.uint32))
    assert np.array_equal(words, oracle.twin_words(
        {lw.LW_FMT_Q4_PAIR: oracle.Q4, lw.LW_FMT_Q6: oracle.Q6, lw.LW_FMT_BF16_EXP: oracle.BF16}[fmt],
        _payload(fmt, m)))
    assert np.array_equal(_host(tw.tensors["tile_off"], np.uint32), ht.view("tile_off", np.uint32))
    assert np.array_equal(_host(tw.tensors["lane_bits"], np.uint16), ht.view("lane_bits", np.uint16))
    assert tw.coded_bytes == ht.stats.coded_bytes


@pytest.mark.parametrize("fmt,make", [CASES[0], CASES[3], CASES[6]])
def test_products_on_the_transcoded_twin(fmt, make):
    m = make()
    db = lw.DeviceBundle.upload(_encode(fmt, m), DEV)
    tw, st = _transcode(db)
    assert st == 0
    B = 3
    x = torch.from_numpy(np.ascontiguousarray(m["x"][:1].repeat(B, 0) *
                                              np.arange(1, B + 1, dtype=np.float32)[:, None])).to(DEV)
    if fmt == lw.LW_FMT_BF16_EXP:
        x = x.to(torch.bfloat16)
    ys = []
    for d, fn in ((db, lw.lw_decode_gemm), (tw, lw.lw_twin_gemm)):
        y = torch.full((B, d.rows), float("nan"), device=DEV)
        ws = torch.zeros(lw.lw_workspace_bytes(d, B) // 4 + 64, device=DEV)
        s = torch.zeros(1, dtype=torch.int32, device=DEV)
        fn(d, x, B, y, ws, s)
        torch.cuda.synchronize()
        assert int(s.item()) == 0
        ys.append(y.cpu().numpy())
    assert np.array_equal(ys[0].view(np.uint32), ys[1].view(np.uint32))


def test_all_verbatim_bf16():
    m = inputs.small_bf16(19, 64, 256, outlier_p=0.5)
    hb, ht = _encode(lw.LW_FMT_BF16_EXP, m), _encode(lw.LW_FMT_BF16_EXP, m, twin=True)
    tw, st = _transcode(lw.DeviceBundle.upload(hb, DEV))
    assert st == 0
    assert np.array_equal(_host(tw.tensors["words"], np.uint32), ht.view("words", np.uint32))


def test_full_size_gate_matrix():
    spec = inputs.workload_specs(inputs.MISTRAL_LAYER)[4]     # gate 14336 x 4096
    m = inputs.make_matrix(inputs.MISTRAL_LAYER, spec, 0, 4)
    hb, ht = _encode(lw.LW_FMT_Q4_PAIR, m), _encode(lw.LW_FMT_Q4_PAIR, m, twin=True)
    tw, st = _transcode(lw.DeviceBundle.upload(hb, DEV))
    assert st == 0
    assert np.array_equal(_host(tw.tensors["words"], np.uint32), ht.view("words", np.uint32))


def test_corrupt_stream_is_reported():
    n, k = 128, 512
    m = inputs.small_q4(5, n, k)
    hb = _encode(lw.LW_FMT_Q4_PAIR, m)
    words = hb.view("words", np.uint32).copy()
    toff = hb.view("tile_off", np.uint32)
    tf = lw.table_fields(hb.sections["table"])
    nsym = np.full((len(toff) - 1, 32), 256, np.int32)
    want = hb.view("lane_bits", np.uint16).reshape(-1, 32)[1, 3]
    for bit in range(31, -1, -1):   # a flip the oracle sees as a wrong lane length
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
    _, st = _transcode(db)
    assert st == 1      # LW_DEV_LANE_LENGTH


def test_bad_views_are_refused():
    m = inputs.small_q4(20, 64, 256)
    db = lw.DeviceBundle.upload(_encode(lw.LW_FMT_Q4_PAIR, m), DEV)
    ht = lw.DeviceBundle.upload(_encode(lw.LW_FMT_Q4_PAIR, m, twin=True), DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    good, _ = _transcode(db)
    import ctypes
    # a twin as the source
    assert lw.load().lw_transcode_twin(ht.ref, good.ref, lw._tp(st), lw._stream_ptr(None)) == \
        lw.LW_ERR_INVALID_ARG
    # wrong max_tile_rows / not a twin / other shape
    for field, val in (("max_tile_rows", 63), ("twin", 0), ("rows", 128), ("fmt", lw.LW_FMT_Q6)):
        v = lw.LwDevBundle.from_buffer_copy(good.view)
        setattr(v, field, val)
        assert lw.load().lw_transcode_twin(db.ref, ctypes.byref(v), lw._tp(st), lw._stream_ptr(None)) != 0
    # twin words on top of the coded words
    v = lw.LwDevBundle.from_buffer_copy(good.view)
    v.words = db.view.words
    assert lw.load().lw_transcode_twin(db.ref, ctypes.byref(v), lw._tp(st), lw._stream_ptr(None)) == \
        lw.LW_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert lw.lw_twin_tile_rows(lw.LW_FMT_Q4_PAIR) == 64
    assert lw.lw_twin_tile_rows(lw.LW_FMT_Q6) == 96
    assert lw.lw_twin_tile_rows(lw.LW_FMT_BF16_EXP) == 64
    assert lw.lw_twin_tile_rows(9) == 0
