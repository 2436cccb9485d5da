"""The oracle's pins are strong enough to catch plausible mistakes.

Each case plants one mistake in the CPU oracle (a monkeypatched function: a
swapped nibble order, the wrong rows in a lane, an off-by-one decoder
quantity, a wrong dequantisation offset, ...) and re-runs every pin of
``test_oracle_pins.py``; at least one pin must fail (an assertion, or an
error raised by the oracle's own checks).
Nothing here touches the library or a GPU.  CPU only."""
import inspect

import numpy as np
import pytest

import oracle
import oracle.oracle as O
import test_oracle_pins as pins


def _pin_calls():
    """Every pin of test_oracle_pins as (name, zero-argument callable),
    parametrised pins expanded over their parameter sets."""
    calls = []
    for name, fn in inspect.getmembers(pins, inspect.isfunction):
        if not name.startswith("test_") or fn.__module__ != pins.__name__:
            continue
        marks = [m for m in getattr(fn, "pytestmark", []) if m.name == "parametrize"]
        if not marks:
            calls.append((name, fn))
            continue
        argnames, values = marks[0].args[0], marks[0].args[1]
        argnames = [a.strip() for a in argnames.split(",")] if isinstance(argnames, str) else list(argnames)
        for v in values:
            v = v if len(argnames) > 1 else (v,)
            kw = dict(zip(argnames, v))
            calls.append((f"{name}{list(kw.values())}", lambda fn=fn, kw=kw: fn(**kw)))
    return calls


def _failing_pins():
    failed = []
    for name, call in _pin_calls():
        try:
            call()
        except pytest.skip.Exception:
            pass
        except (Exception, pytest.fail.Exception) as e:   # an assertion, or the oracle's own checks
            failed.append((name, type(e).__name__))
    return failed


# ---------------------------------------------------------------- mutants

def _swapped_pairs(codes):
    c = codes.astype(np.uint16)
    return (c[:, 0::2] << 4) | c[:, 1::2]


def _lanes_l_l32(a, per_row):            # lane l carries rows l and l + 32
    n = a.shape[0]
    tr, tk = n // 64, a.shape[1] // per_row
    v = a.reshape(tr, 2, 32, tk, per_row).transpose(0, 3, 2, 1, 4)
    return np.ascontiguousarray(v.reshape(tr * tk, 32, 2 * per_row))


def _rows_l_l32(v, n, per_row):
    tr = n // 64
    tk = v.shape[0] // tr
    a = v.reshape(tr, tk, 32, 2, per_row).transpose(0, 3, 2, 1, 4)
    return np.ascontiguousarray(a.reshape(n, tk * per_row))


def _unlimited_lengths(counts, lmax=11):
    counts = np.asarray(counts)
    depth = pins.textbook_huffman_lengths([int(c) for c in counts])
    out = np.zeros(len(counts), dtype=np.uint8)
    for s, l in depth.items():
        out[s] = l
    return out


def _canonical_descending(lengths):      # ties by descending symbol
    L = [int(v) for v in lengths]
    order = sorted((s for s in range(len(L)) if L[s]), key=lambda s: (L[s], -s))
    codes = np.zeros(len(L), dtype=np.uint32)
    code, prev = 0, L[order[0]] if order else 0
    for i, s in enumerate(order):
        if i:
            code = (code + 1) << (L[s] - prev)
        codes[s] = code
        prev = L[s]
    return codes


def _tables_with(key, change):
    def f(lengths, *a, **k):
        t = dict(O_decoder_tables(lengths, *a, **k))
        t[key] = change(np.array(t[key], copy=True))
        return t
    return f


O_decoder_tables = O.decoder_tables


def _limits_unshifted(lim):
    out = lim.copy()
    for l in range(1, len(out)):
        out[l] = out[l] >> (11 - l) if l < 11 else out[l]
    return out


def _fields_sign_bit14(bits):
    b = bits.astype(np.uint16)
    exp = ((b >> 7) & 0xFF).astype(np.uint8)
    sm = (((b >> 7) & 0x80) | (b & 0x7F)).astype(np.uint8)
    return exp, sm


def _palette_top15(exp):
    c = np.bincount(exp.ravel(), minlength=256)
    ranked = sorted((e for e in range(256) if c[e]), key=lambda e: (-int(c[e]), e))
    return np.array(sorted(ranked[:15]), dtype=np.uint8)


def _palette_frequency_order(exp):
    c = np.bincount(exp.ravel(), minlength=256)
    ranked = sorted((e for e in range(256) if c[e]), key=lambda e: (-int(c[e]), e))
    return np.array(ranked[:16], dtype=np.uint8)


def _verbatim_all_outside(exp, palette):  # "every" where the rule says "some"
    inpal = np.isin(exp, palette)
    n, k = exp.shape
    return ~inpal.reshape(n, k // 64, 64).any(axis=2)


def _q4_min_subtracted(codes, scales, mins):
    c = np.asarray(codes, dtype=np.float64)
    s = np.repeat(O.fp16_to_f64(scales), 256, axis=1)
    m = np.repeat(O.fp16_to_f64(mins), 256, axis=1)
    return s * c - m


def _q6_offset_31(codes, scales):
    c = np.asarray(codes, dtype=np.float64)
    return np.repeat(O.fp16_to_f64(scales), 16, axis=1) * (c - 31.0)


O_gemm = O.gemm


def _gemm_drops_last_column(w, x):
    w = np.asarray(w, dtype=np.float64).copy()
    w[:, -1] = 0.0
    return O_gemm(w, x)


O_twin_words = O.twin_words


def _twin_lsb_first(fmt, payload):
    w = O_twin_words(fmt, payload).astype(np.uint64)
    r = np.zeros_like(w)
    for b in range(32):
        r |= ((w >> b) & 1) << (31 - b)
    return r.astype(np.uint32)


O_encode = O.encode


def _encode_mid_from_second_row(fmt, payload):
    out = O_encode(fmt, payload)
    out["lane_mid"] = (out["lane_bits"].astype(np.int64) - out["lane_mid"]).astype(np.uint16)
    return out


O_decode_lanes = O.decode_lanes


def _decode_lanes_shifted(*a, **k):      # every lane's symbols one position late
    out, bits = O_decode_lanes(*a, **k)
    out = np.roll(out, 1, axis=2)
    out[:, :, 0] = 0
    return out, bits


def _join_drops_mantissa_lsb(exp, sm):
    e = exp.astype(np.uint16)
    s = sm.astype(np.uint16)
    return ((s & 0x80) << 8) | (e << 7) | (s & 0x7E)


MUTANTS = {
    "pair nibble order swapped": {"q4_pair_symbols": _swapped_pairs},
    "lane l holds rows l and l+32": {"lanes_from_rows": _lanes_l_l32, "rows_from_lanes": _rows_l_l32},
    "length limit ignored": {"code_lengths": _unlimited_lengths},
    "every code one bit longer": {
        "code_lengths": lambda c, lmax=11, f=O.code_lengths: (lambda L: (L + (L > 0)).astype(L.dtype))(f(c, lmax))},
    "canonical ties by descending symbol": {"canonical_codes": _canonical_descending},
    "decoder base off by one": {"decoder_tables": _tables_with("base", lambda b: b + 1)},
    "limits not left-aligned to 11 bits": {"decoder_tables": _tables_with("limit", _limits_unshifted)},
    "sign bit taken from bit 14": {"bf16_fields": _fields_sign_bit14},
    "palette of 15": {"bf16_palette": _palette_top15},
    "palette in frequency order": {"bf16_palette": _palette_frequency_order},
    "verbatim only when every exponent is outside": {"bf16_verbatim_groups": _verbatim_all_outside},
    "4-bit minimum subtracted": {"dequant_q4": _q4_min_subtracted},
    "6-bit code offset 31": {"dequant_q6": _q6_offset_31},
    "fp16 scales read as bf16": {"fp16_to_f64": O.bf16_to_f64},
    "product drops the last column": {"gemm": _gemm_drops_last_column},
    "twin words LSB-first": {"twin_words": _twin_lsb_first},
    "second-row offset counted from the lane end": {"encode": _encode_mid_from_second_row},
    "decoded symbols one position late": {"decode_lanes": _decode_lanes_shifted},
    "join drops the mantissa's last bit": {"bf16_join": _join_drops_mantissa_lsb},
}


def test_unmutated_oracle_passes_every_pin():
    assert _failing_pins() == []


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_planted_mistake_fails_a_pin(mutant, monkeypatch):
    for name, fn in MUTANTS[mutant].items():
        monkeypatch.setattr(O, name, fn)
        if hasattr(oracle, name):
            monkeypatch.setattr(oracle, name, fn)
    failed = _failing_pins()
    assert failed, f"no pin catches: {mutant}"
    print(mutant, "->", failed)
