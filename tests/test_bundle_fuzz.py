"""Bundle strings are untrusted input: structured mutations of every section
and header field, each re-serialised with consistent section sizes and a
valid checksum so that it reaches the loader's deeper checks.  The loader
must answer every one with LW_OK or a status (LW_ERR_CORRUPT,
LW_ERR_UNSUPPORTED) -- never crash -- and a bundle it accepts must pass
lw_validate_sections again.  CPU only; the mutations are seeded."""
import struct

import numpy as np
import pytest

from decode_gemv_gb300 import inputs
from decode_gemv_gb300 import lw

SECTIONS = lw.SECTION_NAMES
ELEM = {"words": 4, "tile_off": 4, "lane_bits": 2, "table": 1, "qparams": 2, "signman": 1,
        "vflags": 4, "vrow_off": 4, "vexp": 1, "lane_mid": 2}


def fnv1a64(data: bytes) -> int:
    h, mask = 0xcbf29ce484222325, 0xFFFFFFFFFFFFFFFF
    for b in memoryview(data).tolist():
        h = ((h ^ b) * 0x100000001b3) & mask
    return h


def parse(data: bytes):
    head = bytearray(data[:192])
    sizes = struct.unpack_from("<16Q", data, 56)
    secs, off = {}, 192
    for i, name in enumerate(SECTIONS):
        off = (off + 63) // 64 * 64
        secs[name] = bytearray(data[off:off + sizes[i]])
        off += sizes[i]
    return head, secs


def seal(head: bytearray, secs: dict) -> bytes:
    """A bundle string with the header's section sizes set from `secs`, the
    documented 64-byte alignment and a valid checksum."""
    head = bytearray(head)
    for i, name in enumerate(SECTIONS):
        struct.pack_into("<Q", head, 56 + 8 * i, len(secs[name]))
    out = bytearray(head)
    for name in SECTIONS:
        out += b"\0" * ((-len(out)) % 64)
        out += secs[name]
    out += b"\0" * ((-len(out)) % 64)
    return bytes(out) + struct.pack("<Q", fnv1a64(bytes(out)))


def load(data: bytes):
    """LW_OK (and the re-validated bundle) or the refusing status."""
    try:
        hb = lw.lw_bundle_deserialize(data)
    except lw.LwError as e:
        assert e.status in (lw.LW_ERR_CORRUPT, lw.LW_ERR_UNSUPPORTED), e
        return e.status
    lw.lw_validate_sections(hb.desc.fmt, hb.desc.rows, hb.desc.cols, hb.sections,
                            hb.stats.max_tile_rows, twin=hb.twin)
    return lw.LW_OK


def _bundles():
    m4 = inputs.small_q4(21, 128, 512)
    m6 = inputs.small_q6(22, 64, 512)
    mb = inputs.small_bf16(23, 128, 512, outlier_p=0.01)
    out = []
    for twin in (False, True):
        out.append(lw.lw_encode_bundle(lw.LW_FMT_Q4_PAIR, m4["codes"], m4["scales"], m4["mins"],
                                       twin=twin))
        out.append(lw.lw_encode_bundle(lw.LW_FMT_Q6, m6["codes"], m6["scales"], twin=twin))
        out.append(lw.lw_encode_bundle(lw.LW_FMT_BF16_EXP, mb["bits"], twin=twin))
    return out


def mutations(head, secs, rng):
    """(label, head, secs) variants of one bundle."""
    present = [n for n in SECTIONS if len(secs[n])]
    for name in present:
        e, s = ELEM[name], secs[name]
        yield f"{name} minus one element", head, {**secs, name: s[:-e]}
        yield f"{name} halved", head, {**secs, name: s[:len(s) // 2 // e * e]}
        yield f"{name} emptied", head, {**secs, name: bytearray()}
        yield f"{name} plus one element", head, {**secs, name: s + bytearray(rng.bytes(e))}
        for _ in range(4):
            t = bytearray(s)
            k = int(rng.integers(0, len(t)))
            t[k] = int(rng.integers(0, 256))
            yield f"{name} byte {k}", head, {**secs, name: t}
        t = bytearray(rng.bytes(len(s)))
        yield f"{name} random", head, {**secs, name: t}
    for name in ("tile_off", "vrow_off"):
        if not len(secs[name]):
            continue
        v = np.frombuffer(bytes(secs[name]), np.uint32).copy()
        for label, w in (("last huge", np.r_[v[:-1], 0xFFFFFFFF]), ("first nonzero", np.r_[1, v[1:]]),
                         ("decreasing", v[::-1].copy()), ("zeros", np.zeros_like(v)),
                         ("one up", v + np.uint32(1))):
            yield f"{name} {label}", head, {**secs, name: bytearray(w.astype(np.uint32).tobytes())}
    for name in ("lane_bits", "lane_mid"):
        if not len(secs[name]):
            continue
        v = np.frombuffer(bytes(secs[name]), np.uint16).copy()
        for label, w in (("max", np.full_like(v, 0xFFFF)), ("plus 32", v + np.uint16(32))):
            yield f"{name} {label}", head, {**secs, name: bytearray(w.tobytes())}
    for off, fmt_, label in ((16, "<i", "fmt"), (20, "<i", "twin"), (24, "<q", "rows"),
                             (32, "<q", "cols"), (40, "<i", "max_tile_rows"),
                             (44, "<i", "sections"), (48, "<q", "n_verbatim"),
                             (12, "<I", "header bytes"), (184, "<I", "alignment")):
        (v,) = struct.unpack_from(fmt_, head, off)
        for w in (0, -1, v + 1, v - 1, v + 64, v * 2, 1 << 30, -(1 << 31)):
            h = bytearray(head)
            try:
                struct.pack_into(fmt_, h, off, w)
            except struct.error:
                continue
            yield f"header {label} = {w}", h, secs


@pytest.mark.parametrize("index", range(6))
def test_mutated_bundles_are_answered_with_a_status(index):
    hb = _bundles()[index]
    data = lw.lw_bundle_serialize(hb)
    head, secs = parse(data)
    assert load(seal(head, secs)) == lw.LW_OK          # the resealed original loads
    rng = np.random.default_rng(100 + index)
    n, refused = 0, 0
    for label, h, s in mutations(head, secs, rng):
        n += 1
        refused += load(seal(h, s)) != lw.LW_OK
    assert n > 60
    # most structural damage is refused; payload bytes (the coded words, raw
    # sign+mantissa, scales) are not checkable and may load
    assert refused > n // 2


def test_twin_tables_are_checked_too():
    """A twin reads only its table's alphabet and (BF16) palette: both are
    checked on load, so a twin whose palette cannot map indices back to
    exponents in order is refused."""
    for hb in _bundles()[3:]:                     # the three twins
        assert hb.twin
        secs = dict(hb.sections)
        desc = (hb.desc.fmt, hb.desc.rows, hb.desc.cols)

        def validate(table):
            lw.lw_validate_sections(*desc, {**secs, "table": table}, hb.stats.max_tile_rows, twin=True)

        validate(secs["table"])
        t = secs["table"].copy()
        t[4:8] = np.frombuffer(struct.pack("<i", 17), np.uint8)          # alpha
        with pytest.raises(lw.LwError) as e:
            validate(t)
        assert e.value.status == lw.LW_ERR_CORRUPT and "alphabet" in str(e.value)
        if hb.desc.fmt != lw.LW_FMT_BF16_EXP:
            continue
        for n_pal in (0, 17, -1):
            t = secs["table"].copy()
            t[20:24] = np.frombuffer(struct.pack("<i", n_pal), np.uint8)
            with pytest.raises(lw.LwError):
                validate(t)
        t = secs["table"].copy()
        t[896], t[897] = t[897], t[896]                                  # palette order
        with pytest.raises(lw.LwError) as e:
            validate(t)
        assert "ascending" in str(e.value)
