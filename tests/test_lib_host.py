"""liblw host side on the CPU: exports, the bundle builder against the oracle
(cross-decoding, equal optimal size, identical fixed-width twins), tables,
validation and argument errors.  No GPU."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
from decode_gemv_gb300 import inputs
from decode_gemv_gb300 import lw

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    if not os.path.exists(lw.LIB_PATH):
        from decode_gemv_gb300 import build
        build.build()
    lw.load()


def header_functions():
    src = open(os.path.join(ROOT, "include", "lw.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(lw_[a-z0-9_]+)\s*\(", src)))


def test_library_exports_every_declared_function():
    names = header_functions()
    assert len(names) >= 14
    lib = ctypes.CDLL(lw.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(lw.EXPORTED)
    assert lw.load().lw_version() == 4


def _q4(seed, rows, cols, sd=1.6):
    return inputs.small_q4(seed, rows, cols, sd=sd)


@pytest.mark.parametrize("sd", [1.2, 1.6, 2.2])
def test_q4_library_bundle_decodes_with_oracle(sd):
    m = _q4(1, 192, 768, sd)
    hb = lw.lw_encode_bundle(lw.LW_FMT_Q4_PAIR, m["codes"], m["scales"], m["mins"])
    tb = lw.table_fields(hb.sections["table"])
    words = hb.view("words", np.uint32)
    toff = hb.view("tile_off", np.uint32)
    packed = oracle.decode(oracle.Q4, 192, 768, tb["code_len"], words, toff)
    assert np.array_equal(oracle.unpack_q4(packed), m["codes"])
    # both builders are optimal: equal total coded bits
    ob = oracle.encode(oracle.Q4, m["codes"])
    bits_lib = int(hb.view("lane_bits", np.uint16).astype(np.int64).sum())
    bits_or = int(ob["lane_bits"].astype(np.int64).sum())
    assert bits_lib == bits_or
    hist = ob["histogram"]
    assert int((hist * tb["code_len"]).sum()) == bits_or
    # per-lane second-row offsets: the library's code lengths summed over the
    # first row's symbols (lane order from the oracle)
    syms = oracle.lanes_from_rows(oracle.q4_pair_symbols(m["codes"]), 128)
    want_mid = tb["code_len"].astype(np.int64)[syms[:, :, :128]].sum(axis=2)
    assert np.array_equal(hb.view("lane_mid", np.uint16).reshape(-1, 32), want_mid)
    # the oracle's lane bit counts agree with the library's per lane
    _, used = oracle.decode_lanes(tb["code_len"], words, toff, np.full((len(toff) - 1, 32), 256, np.int32), 256)
    assert np.array_equal(used, hb.view("lane_bits", np.uint16).reshape(-1, 32).astype(np.uint32))
    assert tb["lmax"] <= 11


def test_q6_library_bundle_decodes_with_oracle():
    m = inputs.small_q6(2, 128, 512)
    hb = lw.lw_encode_bundle(lw.LW_FMT_Q6, m["codes"], m["scales"])
    tb = lw.table_fields(hb.sections["table"])
    out = oracle.decode(oracle.Q6, 128, 512, tb["code_len"], hb.view("words", np.uint32),
                        hb.view("tile_off", np.uint32))
    assert np.array_equal(out, m["codes"])
    ob = oracle.encode(oracle.Q6, m["codes"])
    assert int(hb.view("lane_bits", np.uint16).astype(np.int64).sum()) == int(ob["lane_bits"].astype(np.int64).sum())


def test_table_matches_oracle_decoder_quantities():
    m = _q4(3, 128, 1024, 1.6)
    hb = lw.lw_encode_bundle(lw.LW_FMT_Q4_PAIR, m["codes"], m["scales"], m["mins"])
    tb = lw.table_fields(hb.sections["table"])
    t = oracle.decoder_tables(tb["code_len"])
    lmin, lmax = tb["lmin"], tb["lmax"]
    for L in range(lmin, lmax + 1):
        assert tb["off"][L - lmin] == int(t["base"][L]) - int(t["first_code"][L])
        if L < lmax:
            assert int(tb["lim_m1"][L - lmin]) == (int(t["limit"][L]) << 21) - 1
    assert list(tb["sym"][: tb["n_sym"]]) == list(t["sorted"])


def test_oracle_bundle_passes_library_validation_and_table_rebuild():
    m = _q4(4, 128, 512, 2.0)
    ob = oracle.encode(oracle.Q4, m["codes"])
    table = lw.lw_table_from_lengths(lw.LW_FMT_Q4_PAIR, ob["code_len"])
    qp = lw.lw_encode_bundle(lw.LW_FMT_Q4_PAIR, m["codes"], m["scales"], m["mins"]).sections["qparams"]
    wt = np.diff(ob["tile_off"]).max()
    secs = dict(words=ob["words"], tile_off=ob["tile_off"], lane_bits=ob["lane_bits"],
                table=table, qparams=qp, lane_mid=ob["lane_mid"])
    lw.lw_validate_sections(lw.LW_FMT_Q4_PAIR, 128, 512, secs, int(wt))
    bad = dict(secs, tile_off=ob["tile_off"].copy())
    bad["tile_off"][3] += 1
    with pytest.raises(lw.LwError) as e:
        lw.lw_validate_sections(lw.LW_FMT_Q4_PAIR, 128, 512, bad, int(wt) + 1)
    assert e.value.status == 5
    bad_table = table.copy()
    bad_table[80] ^= 1      # first per-length offset
    with pytest.raises(lw.LwError):
        lw.lw_validate_sections(lw.LW_FMT_Q4_PAIR, 128, 512, dict(secs, table=bad_table), int(wt))


def test_table_from_lengths_rejects_bad_codes():
    with pytest.raises(lw.LwError):
        lw.lw_table_from_lengths(lw.LW_FMT_Q4_PAIR, [1, 2, 2, 3] + [0] * 252)   # over-full
    with pytest.raises(lw.LwError):
        lw.lw_table_from_lengths(lw.LW_FMT_Q4_PAIR, [2, 2, 2] + [0] * 253)      # incomplete
    with pytest.raises(lw.LwError):
        lw.lw_table_from_lengths(lw.LW_FMT_Q4_PAIR, [12, 1] + [0] * 254)
    t = lw.table_fields(lw.lw_table_from_lengths(lw.LW_FMT_Q4_PAIR, [0, 1] + [0] * 254))
    assert t["phantom"] == 1 and t["n_sym"] == 1 and list(t["sym"][:2]) == [1, 1]


@pytest.mark.parametrize("fmt", [oracle.Q4, oracle.Q6])
def test_twin_words_identical_to_oracle(fmt):
    m = _q4(5, 128, 512) if fmt == oracle.Q4 else inputs.small_q6(5, 128, 512)
    hb = lw.lw_encode_bundle(fmt, m["codes"], m["scales"], m.get("mins"), twin=True)
    assert np.array_equal(hb.view("words", np.uint32), oracle.twin_words(fmt, m["codes"]))
    wt = 64 if fmt == oracle.Q4 else 96
    assert np.array_equal(hb.view("tile_off", np.uint32), np.arange(5, dtype=np.uint32) * wt)


def test_bf16_twin_against_oracle():
    m = inputs.small_bf16(9, 128, 512, outlier_p=0.004)
    hb = lw.lw_encode_bundle(lw.LW_FMT_BF16_EXP, m["bits"], twin=True)
    assert np.array_equal(hb.view("words", np.uint32), oracle.twin_words(oracle.BF16, m["bits"]))
    assert np.array_equal(hb.view("tile_off", np.uint32), np.arange(5, dtype=np.uint32) * 64)
    sp = oracle.bf16_split(m["bits"])
    tb = lw.table_fields(hb.sections["table"])
    assert list(tb["palette"][: tb["n_palette"]]) == list(sp["palette"])
    assert np.array_equal(hb.view("vexp", np.uint8).reshape(-1, 64), sp["vexp"])


def test_q4_qparams_layout():
    m = _q4(6, 128, 768)
    hb = lw.lw_encode_bundle(lw.LW_FMT_Q4_PAIR, m["codes"], m["scales"], m["mins"])
    qp = hb.view("qparams", np.uint16).reshape(-1, 64, 2)
    tk = 3
    for t in range(6):
        s, kt = divmod(t, tk)
        assert np.array_equal(qp[t, :, 0], m["scales"][64 * s: 64 * s + 64, kt])
        assert np.array_equal(qp[t, :, 1], m["mins"][64 * s: 64 * s + 64, kt])


def test_q6_qparams_layout():
    m = inputs.small_q6(7, 64, 512)
    hb = lw.lw_encode_bundle(lw.LW_FMT_Q6, m["codes"], m["scales"])
    qp = hb.view("qparams", np.uint16).reshape(-1, 4, 32, 8)
    for t in range(2):
        for l in (0, 13, 31):
            got = np.concatenate([qp[t, q, l] for q in range(4)])
            want = np.concatenate([m["scales"][2 * l, 16 * t: 16 * t + 16],
                                   m["scales"][2 * l + 1, 16 * t: 16 * t + 16]])
            assert np.array_equal(got, want)


def test_bf16_sections_against_oracle():
    m = inputs.small_bf16(8, 128, 1024, outlier_p=0.004)
    hb = lw.lw_encode_bundle(lw.LW_FMT_BF16_EXP, m["bits"])
    sp = oracle.bf16_split(m["bits"])
    tb = lw.table_fields(hb.sections["table"])
    assert list(tb["palette"][: tb["n_palette"]]) == list(sp["palette"])
    n, k = 128, 1024
    gw = (k // 64 + 31) // 32
    vf = hb.view("vflags", np.uint32).reshape(n, gw)
    flags = np.array([[(vf[r, g // 32] >> (g % 32)) & 1 for g in range(k // 64)] for r in range(n)], bool)
    assert np.array_equal(flags, sp["verbatim"])
    assert np.array_equal(hb.view("vexp", np.uint8).reshape(-1, 64), sp["vexp"])
    vo = hb.view("vrow_off", np.uint32)
    assert vo[-1] == sp["verbatim"].sum()
    # sign+mantissa: byte q of lane l of tile t at t*16384 + ((q/16)*32 + l)*16 + q%16
    sm = hb.view("signman", np.uint8)
    tk = k // 256
    for t, l, q in [(0, 0, 0), (3, 7, 300), (5, 31, 511), (2, 16, 17)]:
        s, kt = divmod(t, tk)
        r = 64 * s + 2 * l + q // 256
        assert sm[t * 16384 + ((q // 16) * 32 + l) * 16 + q % 16] == sp["sm"][r, 256 * kt + q % 256]
    # the coded exponents decode with the oracle
    out = oracle.decode(oracle.BF16, n, k, tb["code_len"][:16], hb.view("words", np.uint32),
                        hb.view("tile_off", np.uint32), palette=sp["palette"],
                        verbatim=sp["verbatim"], vexp=sp["vexp"], sm=sp["sm"])
    assert np.array_equal(out, m["bits"])
    ob = oracle.encode(oracle.BF16, m["bits"])
    assert int(hb.view("lane_bits", np.uint16).astype(np.int64).sum()) == int(ob["lane_bits"].astype(np.int64).sum())
    # second-row offsets: the same wherever the two optimal codes agree on
    # the first row's length (always, if the code lengths coincide)
    if np.array_equal(tb["code_len"][:16], ob["code_len"]):
        assert np.array_equal(hb.view("lane_mid", np.uint16).reshape(-1, 32), ob["lane_mid"])


def test_encode_rejects_bad_arguments():
    with pytest.raises(lw.LwError) as e:
        lw.lw_encode_bundle(lw.LW_FMT_Q4_PAIR, np.zeros((65, 256), np.uint8),
                            np.zeros((65, 1), np.uint16), np.zeros((65, 1), np.uint16))
    assert e.value.status == 2
    with pytest.raises(lw.LwError) as e:
        lw.lw_encode_bundle(lw.LW_FMT_Q4_PAIR, np.full((64, 256), 16, np.uint8),
                            np.zeros((64, 1), np.uint16), np.zeros((64, 1), np.uint16))
    assert e.value.status == 1
    with pytest.raises(lw.LwError) as e:
        lw.lw_encode_bundle(9, np.zeros((64, 256), np.uint8))
    assert e.value.status == 3


def test_single_symbol_and_all_verbatim_bundles():
    z = np.full((64, 256), 3, np.uint8)
    ones = np.zeros((64, 1), np.uint16)
    hb = lw.lw_encode_bundle(lw.LW_FMT_Q4_PAIR, z, ones, ones)
    tb = lw.table_fields(hb.sections["table"])
    assert tb["phantom"] == 1 and hb.stats.max_tile_rows == 8
    r, k = np.indices((64, 256))
    exp = (100 + (r * 7 + k) % 16).astype(np.uint16)
    exp[:, ::64] = 200 + (r[:, ::64] * 4 + k[:, ::64] // 64) % 40
    bits = (exp << 7) | (k % 128).astype(np.uint16)
    hb = lw.lw_encode_bundle(lw.LW_FMT_BF16_EXP, bits)
    assert hb.stats.n_verbatim == 64 * 4 and hb.stats.max_tile_rows == 0


def test_host_calls_from_many_threads():
    """The host builder keeps no shared mutable state: bundles encoded on
    eight threads at once (ctypes releases the interpreter lock during the
    call) are byte-for-byte the ones encoded one after another, and each
    thread's failing call reports its own error text."""
    from concurrent.futures import ThreadPoolExecutor
    mats = [inputs.small_q4(40 + i, 128, 1024, sd=1.2 + 0.1 * i) for i in range(8)]

    def enc(m):
        hb = lw.lw_encode_bundle(lw.LW_FMT_Q4_PAIR, m["codes"], m["scales"], m["mins"])
        return {k: v.tobytes() for k, v in hb.sections.items()}

    want = [enc(m) for m in mats]
    with ThreadPoolExecutor(8) as ex:
        got = list(ex.map(enc, mats * 2))
    assert got == want * 2

    def bad(i):
        codes = np.full((64, 256 * (i + 1)), 16 + i, np.uint8)       # out of range
        try:
            lw.lw_encode_bundle(lw.LW_FMT_Q4_PAIR, codes, np.zeros((64, i + 1), np.uint16),
                                np.zeros((64, i + 1), np.uint16))
        except lw.LwError as e:
            return str(e)
        return ""
    with ThreadPoolExecutor(8) as ex:
        msgs = list(ex.map(bad, range(8)))
    for i, msg in enumerate(msgs):
        assert f"code {16 + i} out of range" in msg, msg


def test_workspace_bytes_follow_the_documented_layout():
    """lw_workspace_bytes = per-strip counters (N/64 uint32, padded to 256
    bytes) + fp32 partial sums [K/256][8][N]; BF16 products of 16 or more
    rows (coded or direct-palette twin) use the tensor-core K-split partials
    [min(max(K/512, 1), 32)][64][N] when larger.  Host arithmetic only: the view's addresses are never used."""
    lib = lw.load()
    for fmt in (lw.LW_FMT_Q4_PAIR, lw.LW_FMT_Q6, lw.LW_FMT_BF16_EXP):
        for n, k in ((64, 256), (192, 768), (4096, 4096), (14336, 4096), (4096, 14336)):
            v = lw.LwDevBundle()
            v.fmt, v.twin, v.rows, v.cols = fmt, 0, n, k
            counters = (n // 64 * 4 + 255) // 256 * 256
            part = (k // 256) * 8 * n * 4
            for batch in (1, 2, 5):
                assert lib.lw_workspace_bytes(ctypes.byref(v), batch) == counters + part
            if fmt == lw.LW_FMT_BF16_EXP:
                splits = min(max(k // 512, 1), 32)
                want = counters + max(part, splits * 64 * n * 4)
                assert lib.lw_workspace_bytes(ctypes.byref(v), 16) == want
                v.twin = 1                      # the direct-palette twin takes the tensor cores too
                assert lib.lw_workspace_bytes(ctypes.byref(v), 16) == want
                assert lib.lw_workspace_bytes(ctypes.byref(v), 5) == counters + part
    v = lw.LwDevBundle()
    v.fmt, v.rows, v.cols = lw.LW_FMT_Q4_PAIR, 64, 256
    assert lib.lw_workspace_bytes(ctypes.byref(v), 0) == 0
    assert lib.lw_workspace_bytes(None, 1) == 0


def test_group_workspace_is_the_members_slices():
    """lw_workspace_bytes_group = the sum over the members of their one-row
    workspace rounded up to 256 bytes (consecutive slices); 0 for an empty,
    oversized or NULL-holding group."""
    lib = lw.load()
    views = []
    for n, k in ((4096, 4096), (1024, 4096), (192, 768)):
        v = lw.LwDevBundle()
        v.fmt, v.rows, v.cols = lw.LW_FMT_Q4_PAIR, n, k
        views.append(v)
    arr = (ctypes.c_void_p * 3)(*[ctypes.addressof(v) for v in views])
    want = sum((lib.lw_workspace_bytes(ctypes.byref(v), 1) + 255) // 256 * 256 for v in views)
    assert lib.lw_workspace_bytes_group(arr, 3) == want
    assert lib.lw_workspace_bytes_group(arr, 0) == 0
    assert lib.lw_workspace_bytes_group(arr, 9) == 0
    arr[1] = None
    assert lib.lw_workspace_bytes_group(arr, 3) == 0
