"""Bundle files (lw_bundle_serialize / _deserialize / _save / _load): the
distribution form of a coded bundle ("Unweight: Compressing LLM Weights for
Faster Inference", "One Format, Two Purposes").

The layout is pinned from outside the library: the header fields are read
back with struct, the sections are found at their documented 64-byte-aligned
offsets and compared byte for byte with lw_bundle_sections, and the checksum
is recomputed here from the FNV-1a definition (offset basis 0xcbf29ce484222325,
prime 0x100000001b3).  A loaded bundle decodes with the oracle to the
original weights.  Corruption anywhere is refused."""
import struct

import numpy as np
import pytest

import oracle
from decode_gemv_gb300 import inputs
from decode_gemv_gb300 import lw

SECTIONS = lw.SECTION_NAMES


def fnv1a64(data: bytes) -> int:
    h = 0xcbf29ce484222325
    for b in data:
        h ^= b
        h = (h * 0x100000001b3) & 0xFFFFFFFFFFFFFFFF
    return h


def fnv1a64_np(data: bytes) -> int:
    """The same hash over a long string (a tight loop over a list)."""
    h = 0xcbf29ce484222325
    mask = 0xFFFFFFFFFFFFFFFF
    for b in memoryview(data).tolist():
        h = ((h ^ b) * 0x100000001b3) & mask
    return h


def _bundles():
    m4 = inputs.small_q4(5, 128, 512)
    m6 = inputs.small_q6(6, 64, 512)
    mb = inputs.small_bf16(7, 128, 512)
    out = []
    for twin in (False, True):
        out.append(("q4", twin, m4, lw.lw_encode_bundle(lw.LW_FMT_Q4_PAIR, m4["codes"], m4["scales"],
                                                        m4["mins"], twin=twin)))
        out.append(("q6", twin, m6, lw.lw_encode_bundle(lw.LW_FMT_Q6, m6["codes"], m6["scales"],
                                                        twin=twin)))
        out.append(("bf16", twin, mb, lw.lw_encode_bundle(lw.LW_FMT_BF16_EXP, mb["bits"], twin=twin)))
    return out


BUNDLES = None


def bundles():
    global BUNDLES
    if BUNDLES is None:
        BUNDLES = _bundles()
    return BUNDLES


def _layout(data: bytes):
    """Parse the documented layout; returns (header dict, {name: bytes}, end)."""
    assert data[:8] == b"LWBUNDLE"
    version, hdr = struct.unpack_from("<II", data, 8)
    fmt, twin, rows, cols = struct.unpack_from("<iiqq", data, 16)
    mtr, nsec, nverb = struct.unpack_from("<iiq", data, 40)
    sizes = struct.unpack_from("<16Q", data, 56)
    align, zero = struct.unpack_from("<II", data, 184)
    head = dict(version=version, header=hdr, fmt=fmt, twin=twin, rows=rows, cols=cols,
                max_tile_rows=mtr, sections=nsec, n_verbatim=nverb, align=align, zero=zero,
                sizes=sizes)
    secs, off = {}, 192
    for i, name in enumerate(SECTIONS):
        off = (off + 63) // 64 * 64
        secs[name] = data[off:off + sizes[i]]
        off += sizes[i]
    end = (off + 63) // 64 * 64
    return head, secs, end


def test_layout_matches_the_documented_format():
    for name, twin, m, hb in bundles():
        data = lw.lw_bundle_serialize(hb)
        head, secs, end = _layout(data)
        assert head["version"] == 1 and head["header"] == 192 and head["align"] == 64
        assert head["zero"] == 0 and head["sections"] == len(SECTIONS)
        assert all(s == 0 for s in head["sizes"][len(SECTIONS):])
        assert (head["fmt"], bool(head["twin"])) == (hb.fmt, twin)
        assert (head["rows"], head["cols"]) == (hb.desc.rows, hb.desc.cols)
        assert head["max_tile_rows"] == hb.stats.max_tile_rows
        assert head["n_verbatim"] == hb.stats.n_verbatim
        for s in SECTIONS:
            want = hb.sections.get(s, np.zeros(0, np.uint8)).tobytes()
            assert secs[s] == want, (name, twin, s)
        assert len(data) == end + 8
        # padding bytes are zero
        mask = bytearray(len(data))
        off = 192
        for i, s in enumerate(SECTIONS):
            off = (off + 63) // 64 * 64
            mask[off:off + head["sizes"][i]] = b"\x01" * head["sizes"][i]
            off += head["sizes"][i]
        pad = [data[i] for i in range(192, end) if not mask[i]]
        assert not any(pad)


def test_checksum_is_fnv1a64_of_everything_before_it():
    for name, twin, m, hb in bundles()[:2]:
        data = lw.lw_bundle_serialize(hb)
        (cks,) = struct.unpack_from("<Q", data, len(data) - 8)
        assert cks == fnv1a64_np(data[:-8])
    # the hash itself against a published test vector of FNV-1a 64
    assert fnv1a64(b"") == 0xcbf29ce484222325
    assert fnv1a64(b"a") == 0xaf63dc4c8601ec8c


def test_round_trip_in_memory_and_through_a_file(tmp_path):
    for name, twin, m, hb in bundles():
        data = lw.lw_bundle_serialize(hb)
        for back in (lw.lw_bundle_deserialize(data), None):
            if back is None:
                p = tmp_path / f"{name}_{int(twin)}.lwb"
                lw.lw_bundle_save(hb, p)
                assert p.read_bytes() == data
                back = lw.lw_bundle_load(p)
            assert (back.fmt, back.twin, back.desc.rows, back.desc.cols) == (hb.fmt, twin, hb.desc.rows,
                                                                             hb.desc.cols)
            assert back.stats == hb.stats
            assert sorted(back.sections) == sorted(hb.sections)
            for s in hb.sections:
                assert np.array_equal(back.sections[s], hb.sections[s]), (name, s)
            assert lw.lw_bundle_serialize(back) == data


def test_loaded_bundles_decode_with_the_oracle(tmp_path):
    for name, twin, m, hb in bundles():
        if twin:
            continue
        p = tmp_path / f"{name}.lwb"
        lw.lw_bundle_save(hb, p)
        back = lw.lw_bundle_load(p)
        tb = lw.table_fields(back.sections["table"])
        n, k = back.desc.rows, back.desc.cols
        words, toff = back.view("words", np.uint32), back.view("tile_off", np.uint32)
        if name == "q4":
            out = oracle.unpack_q4(oracle.decode(oracle.Q4, n, k, tb["code_len"], words, toff))
            assert np.array_equal(out, m["codes"])
        elif name == "q6":
            assert np.array_equal(oracle.decode(oracle.Q6, n, k, tb["code_len"], words, toff), m["codes"])
        else:
            sp = oracle.bf16_split(m["bits"])
            out = oracle.decode(oracle.BF16, n, k, tb["code_len"][:16], words, toff,
                                palette=sp["palette"], verbatim=sp["verbatim"], vexp=sp["vexp"],
                                sm=sp["sm"])
            assert np.array_equal(out, m["bits"])


def _reseal(buf: bytearray) -> bytes:
    """Recompute the checksum after an edit (to reach the deeper checks)."""
    struct.pack_into("<Q", buf, len(buf) - 8, fnv1a64_np(bytes(buf[:-8])))
    return bytes(buf)


def _refused(data: bytes, code: int):
    with pytest.raises(lw.LwError) as e:
        lw.lw_bundle_deserialize(data)
    assert e.value.status == code, lw.STATUS_NAMES.get(e.value.status)


def test_corruption_is_refused():
    name, twin, m, hb = bundles()[0]          # 4-bit, coded
    data = lw.lw_bundle_serialize(hb)
    head, secs, end = _layout(data)
    corrupt = lw.LW_ERR_CORRUPT
    # any flipped byte fails the checksum
    rng = np.random.default_rng(0)
    for pos in list(rng.integers(0, len(data), 12)) + [0, 9, 20, 60, 191, len(data) - 1]:
        b = bytearray(data)
        b[int(pos)] ^= 0x10
        with pytest.raises(lw.LwError) as e:
            lw.lw_bundle_deserialize(bytes(b))
        assert e.value.status in (corrupt, lw.LW_ERR_UNSUPPORTED)
    # truncated / extended
    _refused(data[:-1], corrupt)
    _refused(data + b"\0", corrupt)
    _refused(data[:100], corrupt)
    # another version
    b = bytearray(data)
    struct.pack_into("<I", b, 8, 2)
    _refused(_reseal(b), lw.LW_ERR_UNSUPPORTED)
    # resealed but inconsistent: a tile offset that decreases
    b = bytearray(data)
    off = 192
    for i, s in enumerate(SECTIONS):
        off = (off + 63) // 64 * 64
        if s == "tile_off":
            struct.pack_into("<I", b, off + 8, 0xFFFF)
            break
        off += head["sizes"][i]
    _refused(_reseal(b), corrupt)
    # resealed but the header's statistics lie
    b = bytearray(data)
    struct.pack_into("<i", b, 40, head["max_tile_rows"] + 1)
    _refused(_reseal(b), corrupt)
    # resealed with a shape that does not match the sections
    b = bytearray(data)
    struct.pack_into("<q", b, 24, head["rows"] + 64)
    _refused(_reseal(b), corrupt)
    # a table that does not match its code lengths
    b = bytearray(data)
    off = 192
    for i, s in enumerate(SECTIONS):
        off = (off + 63) // 64 * 64
        if s == "table":
            b[off + 32 + 4 * 12] ^= 1        # off[0]
            break
        off += head["sizes"][i]
    _refused(_reseal(b), corrupt)
    # not a bundle at all
    _refused(b"x" * 300, corrupt)


def test_file_errors(tmp_path):
    with pytest.raises(lw.LwError) as e:
        lw.lw_bundle_load(tmp_path / "missing.lwb")
    assert e.value.status == lw.LW_ERR_IO
    name, twin, m, hb = bundles()[0]
    with pytest.raises(lw.LwError) as e:
        lw.lw_bundle_save(hb, tmp_path / "no_such_dir" / "x.lwb")
    assert e.value.status == lw.LW_ERR_IO
