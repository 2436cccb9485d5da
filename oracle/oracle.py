"""CPU oracle for entropy-coded weights -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this module.  The product library never calls it and shares no
code with it.  Bit-level work (package-merge, canonical codes, lane packing,
comparator decoding, the fp64 dot products) lives in ``lw_oracle.c``; this file
builds that with gcc on first use and arranges symbols into lanes with plain
numpy reshapes.

What each function follows is cited in its docstring.  Sources:

* "LazyWeights: Decode-on-Demand Edge LLMs" (page 1): sections "2 . Code
  them", "3 . Decode on demand", Fig. 3(a)/(b).
* "Unweight: Compressing LLM Weights for Faster Inference" (page 2):
  "Understanding BF16 weight structure", "The exponent's exploitable
  redundancy" (top-16 palette, raw sign+mantissa, verbatim rows of 64).
* "Software-Defined Bandwidth Expansion" (page 3): section IV.A (grouped
  low-bit storage, codec idempotence on its lattice), eq. (1) (B_eff).

Readings taken where the pages are silent:
tile = 64 rows x 256 columns; lane l holds rows 2l and 2l+1, row 2l first,
columns ascending; pair symbol = c[k] | c[k+1] << 4 for even k; codes MSB-first
in 32-bit words; lanes zero-padded to the tile's longest lane; package-merge
lengths; RFC 1951 canonical order; BF16 palette = 16 most frequent exponents
(ties to the smaller value), indexed in ascending exponent order; a "row of 64"
is 64 consecutive columns of one matrix row.

Parity pins: every function here is pinned by a ``-m "not gpu"`` test in
``tests/test_oracle_pins.py`` (brute force, closed forms, invariants,
exhaustive search, an RFC 1951 example); none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

MAXLEN = 11
Q4, Q6, BF16 = 1, 2, 3
_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "_build", "liblw_oracle.so")
_lib = None
_lock = threading.Lock()


def build() -> str:
    """Compile lw_oracle.c with gcc (plain C, no architecture flags)."""
    os.makedirs(os.path.dirname(_SO), exist_ok=True)
    src = os.path.join(_HERE, "lw_oracle.c")
    tmp = _SO + f".{os.getpid()}.tmp"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-shared", "-fPIC",
                           "-o", tmp, src])
    os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        src = os.path.join(_HERE, "lw_oracle.c")
        if not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(src):
            build()
        lib = ctypes.CDLL(_SO)
        P = ctypes.c_void_p
        i64, i32 = ctypes.c_int64, ctypes.c_int
        lib.or_code_lengths.argtypes = [P, i32, i32, P]
        lib.or_canonical_codes.argtypes = [P, i32, P]
        lib.or_decoder_tables.argtypes = [P, i32, P, P, P, P, P]
        lib.or_pack_lanes.argtypes = [P, i32, P, P, i64, i32, P, P, P]
        lib.or_decode_lanes.argtypes = [P, i32, P, P, i64, P, i32, P, P]
        lib.or_gemm_f64.argtypes = [P, P, i64, i64, i32, P]
        lib.or_gemm_f64.restype = None
        _lib = lib
        return lib


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


# --------------------------------------------------------------------------
# Huffman code construction
# --------------------------------------------------------------------------

def code_lengths(counts, lmax: int = MAXLEN) -> np.ndarray:
    """Optimal prefix-code lengths, none longer than ``lmax`` (package-merge).

    LazyWeights, "2 . Code them": one length-limited Huffman table per matrix
    with 11-bit codes.  Zero-count symbols get no code; a lone symbol gets
    length 1.
    """
    c = np.ascontiguousarray(counts, dtype=np.uint64)
    out = np.zeros(len(c), dtype=np.uint8)
    rc = _load().or_code_lengths(_p(c), len(c), lmax, _p(out))
    if rc:
        raise ValueError(f"or_code_lengths failed ({rc})")
    return out


def canonical_codes(lengths) -> np.ndarray:
    """Canonical code values (RFC 1951 section 3.2.2 rule)."""
    ln = np.ascontiguousarray(lengths, dtype=np.uint8)
    out = np.zeros(len(ln), dtype=np.uint32)
    if _load().or_canonical_codes(_p(ln), len(ln), _p(out)):
        raise ValueError("bad lengths")
    return out


def decoder_tables(lengths) -> dict:
    """first_code, count, limit (11-bit, left-aligned), base, canonical symbol
    order, for L = 0..11 -- the quantities the comparator decoder of
    LazyWeights "3 . Decode on demand" / Fig. 3(b) uses."""
    ln = np.ascontiguousarray(lengths, dtype=np.uint8)
    f, c, lim, b = (np.zeros(MAXLEN + 1, dtype=np.uint32) for _ in range(4))
    srt = np.zeros(len(ln), dtype=np.uint16)
    if _load().or_decoder_tables(_p(ln), len(ln), _p(f), _p(c), _p(lim), _p(b), _p(srt)):
        raise ValueError("bad lengths")
    return dict(first_code=f, count=c, limit=lim, base=b,
                sorted=srt[: int(c.sum())])


# --------------------------------------------------------------------------
# Symbols in lane order
# --------------------------------------------------------------------------

def tile_grid(rows: int, cols: int):
    """(tile rows, tile columns) of a matrix cut into 64 x 256 tiles (a
    reading: LazyWeights "2 . Code them" and Fig. 3(a) code a matrix in
    independently decodable tiles of 32 lanes but fix no tile shape)."""
    if rows % 64 or cols % 256 or rows <= 0 or cols <= 0:
        raise ValueError("shape must be a positive multiple of 64 x 256")
    return rows // 64, cols // 256


def q4_pair_symbols(codes: np.ndarray) -> np.ndarray:
    """Two 4-bit codes -> one 8-bit symbol, even column in the low nibble
    (LazyWeights "2 . Code them": 4-bit codes are coded in pairs)."""
    c = codes.astype(np.uint16)
    return c[:, 0::2] | (c[:, 1::2] << 4)


def lanes_from_rows(a: np.ndarray, per_row: int) -> np.ndarray:
    """[N][TK*per_row] row-major symbols -> [n_tiles][32][2*per_row].

    Tile t = s*TK + kt covers rows 64s..64s+63; lane l carries row 64s+2l then
    row 64s+2l+1, each over the tile's columns in ascending order (LazyWeights
    Fig. 3(a): one Huffman stream per lane, 32 lanes per tile; the rows a lane
    carries are a reading).
    """
    n = a.shape[0]
    tr, tk = n // 64, a.shape[1] // per_row
    v = a.reshape(tr, 32, 2, tk, per_row).transpose(0, 3, 1, 2, 4)
    return np.ascontiguousarray(v.reshape(tr * tk, 32, 2 * per_row))


def rows_from_lanes(v: np.ndarray, n: int, per_row: int) -> np.ndarray:
    """Inverse of lanes_from_rows: [n_tiles][32][2*per_row] -> [N][TK*per_row]
    (the lane-to-row map of LazyWeights Fig. 3(a), read backwards)."""
    tr = n // 64
    tk = v.shape[0] // tr
    a = v.reshape(tr, tk, 32, 2, per_row).transpose(0, 2, 3, 1, 4)
    return np.ascontiguousarray(a.reshape(n, tk * per_row))


# --------------------------------------------------------------------------
# BF16: exponent palette, verbatim groups, sign+mantissa bytes
# --------------------------------------------------------------------------

def bf16_fields(bits: np.ndarray):
    """Split bf16 bit patterns into the exponent byte and the sign+mantissa
    byte (Unweight, "Understanding BF16 weight structure": 1 sign bit, 8
    exponent bits, 7 mantissa bits).  sm = sign << 7 | mantissa."""
    b = bits.astype(np.uint16)
    exp = ((b >> 7) & 0xFF).astype(np.uint8)
    sm = (((b >> 8) & 0x80) | (b & 0x7F)).astype(np.uint8)
    return exp, sm


def bf16_join(exp: np.ndarray, sm: np.ndarray) -> np.ndarray:
    """Inverse of bf16_fields: exponent byte + sign/mantissa byte -> bf16
    bits (Unweight, "Understanding BF16 weight structure")."""
    e = exp.astype(np.uint16)
    s = sm.astype(np.uint16)
    return ((s & 0x80) << 8) | (e << 7) | (s & 0x7F)


def bf16_palette(exp: np.ndarray) -> np.ndarray:
    """The 16 most frequent exponent values of the matrix (ties: the smaller
    value wins), returned in ascending order; fewer if fewer occur.
    Unweight, "The exponent's exploitable redundancy": top-16 palette."""
    counts = np.bincount(exp.ravel(), minlength=256)
    present = [e for e in range(256) if counts[e] > 0]
    ranked = sorted(present, key=lambda e: (-int(counts[e]), e))
    return np.array(sorted(ranked[:16]), dtype=np.uint8)


def bf16_verbatim_groups(exp: np.ndarray, palette: np.ndarray) -> np.ndarray:
    """bool [N][K/64]: True where some exponent of the 64-column group lies
    outside the palette (Unweight: the whole row of 64 is stored verbatim)."""
    inpal = np.isin(exp, palette)
    n, k = exp.shape
    return ~inpal.reshape(n, k // 64, 64).all(axis=2)


def bf16_split(bits: np.ndarray) -> dict:
    """Everything the BF16 path stores besides the coded indices: exponent
    and sign+mantissa bytes, the top-16 palette, the verbatim 64-column
    groups with their raw exponents, and each weight's palette index
    (Unweight, "The exponent's exploitable redundancy")."""
    exp, sm = bf16_fields(bits)
    pal = bf16_palette(exp)
    verb = bf16_verbatim_groups(exp, pal)
    lut = np.full(256, 255, dtype=np.uint8)
    lut[pal] = np.arange(len(pal), dtype=np.uint8)
    idx = lut[exp]                      # palette index (255 = not in palette)
    n, k = exp.shape
    vexp = exp.reshape(n, k // 64, 64)[verb]          # [n_verbatim][64], row-major
    return dict(exp=exp, sm=sm, palette=pal, verbatim=verb, index=idx, vexp=vexp)


def bf16_lane_symbols(index: np.ndarray, verbatim: np.ndarray):
    """Palette indices in lane order, skipping verbatim groups.

    Lane l of a tile walks row 2l then 2l+1 (the lane map of LazyWeights
    Fig. 3(a)); within a row the four 64-column groups in ascending order; a
    verbatim group contributes no symbol (Unweight, "The exponent's
    exploitable redundancy": such rows of 64 bypass the code).
    Returns syms [n_tiles][32][512] (tail unused) and nsym [n_tiles][32].
    """
    n, k = index.shape
    lanes = lanes_from_rows(index, 256).reshape(-1, 32, 8, 64)
    vl = lanes_from_rows(verbatim, 4).reshape(-1, 32, 8)
    order = np.argsort(vl, axis=2, kind="stable")    # coded groups first, in order
    lanes = np.take_along_axis(lanes, order[..., None], axis=2)
    nsym = (64 * (8 - vl.sum(axis=2))).astype(np.int32)
    return np.ascontiguousarray(lanes.reshape(-1, 32, 512).astype(np.uint16)), nsym


# --------------------------------------------------------------------------
# Encode / decode whole matrices
# --------------------------------------------------------------------------

def _symbols(fmt: int, payload: np.ndarray):
    n, k = payload.shape
    tile_grid(n, k)
    if fmt == Q4:
        syms = lanes_from_rows(q4_pair_symbols(payload), 128)
        nsym = np.full(syms.shape[:2], 256, dtype=np.int32)
        return syms.astype(np.uint16), nsym, 256, None
    if fmt == Q6:
        syms = lanes_from_rows(payload.astype(np.uint16), 256)
        nsym = np.full(syms.shape[:2], 512, dtype=np.int32)
        return syms.astype(np.uint16), nsym, 64, None
    if fmt == BF16:
        sp = bf16_split(payload)
        syms, nsym = bf16_lane_symbols(sp["index"], sp["verbatim"])
        return syms, nsym, 16, sp
    raise ValueError("fmt")


def encode(fmt: int, payload: np.ndarray) -> dict:
    """Build the coded sections of one matrix: one length-limited Huffman
    code over the matrix's symbol histogram, each lane's codes packed
    MSB-first into 32-bit words interleaved across the tile's 32 lanes, and
    per-tile word offsets (LazyWeights "2 . Code them", Fig. 3(a)).

    payload: uint8 codes [N][K] (4- or 6-bit) or uint16 bf16 bits [N][K].
    Returns code_len, words, tile_off, lane_bits (+ BF16 side data).
    """
    syms, nsym, alpha, sp = _symbols(fmt, payload)
    maxsym = syms.shape[2]
    coded = np.arange(maxsym)[None, None, :] < nsym[:, :, None]
    used = np.bincount(syms[coded], minlength=alpha).astype(np.uint64)  # histogram
    length = code_lengths(used)
    n_tiles = syms.shape[0]
    lib = _load()
    tile_off = np.zeros(n_tiles + 1, dtype=np.uint32)
    lane_bits = np.zeros((n_tiles, 32), dtype=np.uint16)
    rc = lib.or_pack_lanes(_p(length), alpha, _p(syms), _p(nsym), n_tiles, maxsym,
                           _p(tile_off), _p(lane_bits), None)
    if rc:
        raise ValueError(f"pack failed {rc}")
    words = np.zeros(int(tile_off[-1]) * 32, dtype=np.uint32)
    rc = lib.or_pack_lanes(_p(length), alpha, _p(syms), _p(nsym), n_tiles, maxsym,
                           _p(tile_off), _p(lane_bits), _p(words))
    if rc:
        raise ValueError(f"pack failed {rc}")
    # bit offset where each lane's second row starts: the code lengths of the
    # symbols of its first row, summed
    if fmt == Q4:
        first = np.full(nsym.shape, 128)
    elif fmt == Q6:
        first = np.full(nsym.shape, 256)
    else:
        vl = lanes_from_rows(sp["verbatim"], 4).reshape(-1, 32, 8)
        first = 64 * (4 - vl[:, :, :4].sum(axis=2))
    in_first = np.arange(maxsym)[None, None, :] < first[:, :, None]
    lane_mid = (length.astype(np.int64)[np.where(in_first, syms, 0)] * in_first).sum(axis=2)
    lane_mid = lane_mid.astype(np.uint16)
    out = dict(fmt=fmt, rows=payload.shape[0], cols=payload.shape[1], code_len=length,
               words=words, tile_off=tile_off, lane_bits=lane_bits, lane_mid=lane_mid,
               nsym=nsym, histogram=used)
    if sp is not None:
        out.update(palette=sp["palette"], verbatim=sp["verbatim"], vexp=sp["vexp"],
                   sm=sp["sm"])
    return out


def decode_lanes(code_len, words, tile_off, nsym, maxsym):
    """Comparator decode of every lane (LazyWeights "3 . Decode on demand").
    Returns symbols [n_tiles][32][maxsym] and bits consumed [n_tiles][32]."""
    code_len = np.ascontiguousarray(code_len, dtype=np.uint8)
    words = np.ascontiguousarray(words, dtype=np.uint32)
    tile_off = np.ascontiguousarray(tile_off, dtype=np.uint32)
    nsym = np.ascontiguousarray(nsym, dtype=np.int32)
    n_tiles = len(tile_off) - 1
    out = np.zeros((n_tiles, 32, maxsym), dtype=np.uint16)
    bits = np.zeros((n_tiles, 32), dtype=np.uint32)
    rc = _load().or_decode_lanes(_p(code_len), len(code_len), _p(words), _p(tile_off),
                                 n_tiles, _p(nsym), maxsym, _p(out), _p(bits))
    if rc:
        raise ValueError(f"corrupt stream ({rc})")
    return out, bits


def decode(fmt: int, rows: int, cols: int, code_len, words, tile_off,
           palette=None, verbatim=None, vexp=None, sm=None):
    """Restore the fixed-width payload from the coded sections (LazyWeights
    "3 . Decode on demand"; BF16 exponents through the palette and the
    verbatim groups of Unweight, "The exponent's exploitable redundancy").

    Q4 -> packed bytes [N][K/2] (low nibble = even column), Q6 -> uint8
    [N][K], BF16 -> uint16 bits [N][K].
    """
    tr, tk = tile_grid(rows, cols)
    if fmt == Q4:
        nsym = np.full((tr * tk, 32), 256, dtype=np.int32)
        s, _ = decode_lanes(code_len, words, tile_off, nsym, 256)
        return rows_from_lanes(s, rows, 128).astype(np.uint8)
    if fmt == Q6:
        nsym = np.full((tr * tk, 32), 512, dtype=np.int32)
        s, _ = decode_lanes(code_len, words, tile_off, nsym, 512)
        return rows_from_lanes(s, rows, 256).astype(np.uint8)
    # BF16: re-insert verbatim groups, then map palette index -> exponent
    vl = lanes_from_rows(verbatim, 4).reshape(-1, 32, 8)
    nsym = (64 * (8 - vl.sum(axis=2))).astype(np.int32)
    s, _ = decode_lanes(code_len, words, tile_off, nsym, 512)
    idx = np.zeros((tr * tk, 32, 8, 64), dtype=np.uint16)
    for t in range(tr * tk):
        for l in range(32):
            g_coded = [g for g in range(8) if not vl[t, l, g]]
            for j, g in enumerate(g_coded):
                idx[t, l, g] = s[t, l, 64 * j: 64 * j + 64]
    idx_rows = rows_from_lanes(idx.reshape(-1, 32, 512), rows, 256)
    exp = np.asarray(palette, dtype=np.uint8)[np.minimum(idx_rows, len(palette) - 1)]
    exp = exp.reshape(rows, cols // 64, 64)
    exp[verbatim] = vexp
    return bf16_join(exp.reshape(rows, cols), sm)


def unpack_q4(packed: np.ndarray) -> np.ndarray:
    """Packed 4-bit bytes [N][K/2] -> codes [N][K], low nibble = even column
    (the pair order of q4_pair_symbols)."""
    out = np.empty((packed.shape[0], packed.shape[1] * 2), dtype=np.uint8)
    out[:, 0::2] = packed & 15
    out[:, 1::2] = packed >> 4
    return out


# --------------------------------------------------------------------------
# Dequantisation and products (fp64)
# --------------------------------------------------------------------------

def fp16_to_f64(bits) -> np.ndarray:
    """IEEE binary16 bit patterns -> exact fp64 values (the stored scales
    and minimums)."""
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def bf16_to_f64(bits) -> np.ndarray:
    """bf16 bit patterns -> exact fp64 values (bf16 is the top half of an
    fp32; Unweight, "Understanding BF16 weight structure")."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def dequant_q4(codes, scales, mins) -> np.ndarray:
    """w = scale * code + min, one fp16 scale and min per 256-weight
    super-block of a row (the tiny 4-bit workload's rule; LazyWeights "2 .
    Code them": scales and minimums stay as stored).  Exact in fp64."""
    c = np.asarray(codes, dtype=np.float64)
    s = np.repeat(fp16_to_f64(scales), 256, axis=1)
    m = np.repeat(fp16_to_f64(mins), 256, axis=1)
    return s * c + m


def dequant_q6(codes, scales) -> np.ndarray:
    """w = scale * (code - 32), one fp16 scale per 16 weights of a row
    (Q6_K's code offset; LazyWeights "1 . Select the codes" names llama.cpp's
    Q6_K block format but prints no formula, so this is a reading)."""
    c = np.asarray(codes, dtype=np.float64)
    s = np.repeat(fp16_to_f64(scales), 16, axis=1)
    return s * (c - 32.0)


def gemm(w: np.ndarray, x: np.ndarray) -> np.ndarray:
    """Y[b][r] = sum_k W[r][k] * X[b][k] in fp64, k ascending (plain loops in
    C): the matrix-vector product of LazyWeights "3 . Decode on demand", one
    row of X per batch entry.  Shapes: W [N][K], X [B][K] -> Y [B][N]."""
    w = np.ascontiguousarray(w, dtype=np.float64)
    x = np.ascontiguousarray(np.atleast_2d(x), dtype=np.float64)
    n, k = w.shape
    y = np.zeros((x.shape[0], n), dtype=np.float64)
    _load().or_gemm_f64(_p(w), _p(x), n, k, x.shape[0], _p(y))
    return y


def reference_output(fmt: int, m: dict) -> np.ndarray:
    """Y = deq(W) X for one generated matrix (fp64)."""
    if fmt == Q4:
        return gemm(dequant_q4(m["codes"], m["scales"], m["mins"]), m["x"])
    if fmt == Q6:
        return gemm(dequant_q6(m["codes"], m["scales"]), m["x"])
    return gemm(bf16_to_f64(m["bits"]), bf16_to_f64(m["x"]))


def abs_row_products(fmt: int, m: dict) -> np.ndarray:
    """sum_k |w_rk x_k| per output in fp64: the scale of the componentwise
    check (the standard bound on a floating-point dot product's rounding
    error is proportional to this sum, not to |y|)."""
    if fmt == Q4:
        w = dequant_q4(m["codes"], m["scales"], m["mins"])
        x = m["x"]
    elif fmt == Q6:
        w = dequant_q6(m["codes"], m["scales"])
        x = m["x"]
    else:
        w = bf16_to_f64(m["bits"])
        x = bf16_to_f64(m["x"])
    return gemm(np.abs(w), np.abs(np.atleast_2d(np.asarray(x, dtype=np.float64))))


# --------------------------------------------------------------------------
# Fixed-width twin layout (same tiles, lanes and interleave, no coding)
# --------------------------------------------------------------------------

def twin_words(fmt: int, payload: np.ndarray) -> np.ndarray:
    """Fixed-width twin streams: each lane's values at a constant width (4-bit
    codes / 6-bit codes / 4-bit palette index for BF16), MSB-first in 32-bit
    words, word-interleaved across the tile's 32 lanes (LazyWeights: the
    decode-free "twin" of the same layout)."""
    n, k = payload.shape
    if fmt == Q4:
        lanes, width = lanes_from_rows(payload.astype(np.uint32), 256), 4
    elif fmt == Q6:
        lanes, width = lanes_from_rows(payload.astype(np.uint32), 256), 6
    else:
        sp = bf16_split(payload)
        idx = np.where(sp["index"] == 255, 0, sp["index"]).astype(np.uint32)
        idx = idx.reshape(n, k // 64, 64)
        idx[sp["verbatim"]] = 0
        lanes, width = lanes_from_rows(idx.reshape(n, k), 256), 4
    nt = lanes.shape[0]
    nbits = 512 * width
    bits = np.zeros((nt, 32, nbits), dtype=np.uint8)
    for b in range(width):           # bit b of value i -> stream bit i*width + (width-1-b)
        bits[:, :, (width - 1 - b)::width] = (lanes >> b) & 1
    w = np.packbits(bits.reshape(nt, 32, nbits // 32, 32), axis=3, bitorder="big")
    w = w.view(">u4").reshape(nt, 32, nbits // 32).astype(np.uint32)
    return np.ascontiguousarray(w.transpose(0, 2, 1)).ravel()
