"""rANS — the entropy coder the LazyWeights page weighs Huffman against
("LazyWeights: Decode-on-Demand Edge LLMs", "Decoder hardware", paragraph
"Huffman over rANS": rANS is never smaller, 0.0 to +1.0 % more bits).

TEST AND ANALYSIS INFRASTRUCTURE, like the rest of oracle/: nothing in the
library uses it.  It codes exactly the symbols the Huffman lanes code (one
stream per lane: row 2l's symbols, then row 2l+1's, taken from oracle's
lane split), so the two coders are compared symbol for symbol.

The coder is the textbook byte-renormalising range variant of asymmetric
numeral systems (Duda): a state x in [L, 256 L), L = 2^23; symbol s with
quantised frequency f_s and cumulative start c_s out of M = 2^PREC;
encoding runs over the stream backwards,
    while x >= ((L >> PREC) << 8) * f_s: emit the low byte of x, x >>= 8
    x = (x // f_s) * M + (x mod f_s) + c_s
and ends by emitting the 4 bytes of x; decoding reads x first, then per
symbol: slot = x mod M, s = the symbol whose [c_s, c_s + f_s) holds slot,
x = f_s * (x // M) + slot - c_s, and while x < L: x = 256 x + next byte.
"""
from __future__ import annotations

import numpy as np

PREC = 12
M = 1 << PREC
L = 1 << 23


def quantize(counts, prec: int = PREC) -> np.ndarray:
    """Frequencies out of 2^prec, proportional to counts: every symbol that
    occurs gets at least 1, others 0; largest remainders take the rounding
    slack; a deficit is taken from the largest frequencies."""
    counts = np.asarray(counts, dtype=np.float64)
    total = counts.sum()
    m = 1 << prec
    used = counts > 0
    if used.sum() == 0:
        raise ValueError("no symbols")
    if used.sum() > m:
        raise ValueError("alphabet larger than the frequency total")
    exact = counts * m / total
    f = np.floor(exact).astype(np.int64)
    f[used & (f == 0)] = 1
    rest = m - int(f.sum())
    if rest > 0:
        order = np.argsort(-(exact - np.floor(exact)) * used, kind="stable")
        for i in order[:rest]:
            f[i] += 1
    while rest < 0:
        i = int(np.argmax(f))
        take = min(-rest, int(f[i]) - 1)
        f[i] -= take
        rest += take
    assert f.sum() == m and np.all(f[used] >= 1) and np.all(f[~used] == 0)
    return f


def _cum(freq: np.ndarray) -> np.ndarray:
    return np.concatenate([[0], np.cumsum(freq)[:-1]]).astype(np.int64)


def encode_stream(syms, freq) -> bytes:
    """One stream, plain Python (the definition)."""
    cum = _cum(freq)
    x = L
    out = []
    for s in reversed([int(v) for v in syms]):
        f, c = int(freq[s]), int(cum[s])
        if f == 0:
            raise ValueError(f"symbol {s} has frequency 0")
        x_max = ((L >> PREC) << 8) * f
        while x >= x_max:
            out.append(x & 0xFF)
            x >>= 8
        x = (x // f) * M + (x % f) + c
    for _ in range(4):
        out.append(x & 0xFF)
        x >>= 8
    return bytes(reversed(out))


def decode_stream(data: bytes, n: int, freq) -> np.ndarray:
    cum = _cum(freq)
    slot_sym = np.repeat(np.arange(len(freq)), freq)
    x = int.from_bytes(data[:4], "big")
    pos = 4
    out = np.zeros(n, dtype=np.int64)
    for i in range(n):
        slot = x & (M - 1)
        s = int(slot_sym[slot])
        out[i] = s
        x = int(freq[s]) * (x >> PREC) + slot - int(cum[s])
        while x < L:
            x = (x << 8) | data[pos]
            pos += 1
    if pos != len(data) or x != L:
        raise ValueError("stream not consumed exactly")
    return out


def stream_bytes(syms: np.ndarray, nsym: np.ndarray, freq) -> np.ndarray:
    """Bytes of every stream (final state included), all streams at once:
    syms [S][maxsym] (the first nsym[i] of row i are coded), the same
    arithmetic as encode_stream applied to each stream."""
    syms = np.asarray(syms, dtype=np.int64)
    nsym = np.asarray(nsym, dtype=np.int64)
    freq = np.asarray(freq, dtype=np.int64)
    cum = _cum(freq)
    x = np.full(syms.shape[0], L, dtype=np.int64)
    nbytes = np.full(syms.shape[0], 4, dtype=np.int64)
    for j in range(syms.shape[1] - 1, -1, -1):
        act = j < nsym
        s = np.where(act, syms[:, j], 0)        # past nsym: padding, not coded
        f = np.where(act, freq[s], 1)
        c = cum[s]
        x_max = ((L >> PREC) << 8) * f
        while True:
            over = act & (x >= x_max)
            if not over.any():
                break
            nbytes += over
            x = np.where(over, x >> 8, x)
        x = np.where(act, (x // f) * M + (x % f) + c, x)
    return nbytes


def compare(fmt: int, payload: np.ndarray) -> dict:
    """Huffman lanes (the oracle's optimal 11-bit code) against rANS lanes
    over the same symbols, plus the Shannon bound of the symbol histogram.
    Bits exclude the per-matrix table; Huffman bits are the exact lane bit
    counts (no word or tile padding)."""
    from .oracle import BF16, _symbols, encode
    syms, nsym, alpha, _ = _symbols(fmt, payload)
    enc = encode(fmt, payload)
    hist = enc["histogram"].astype(np.float64)
    p = hist[hist > 0] / hist.sum()
    entropy_bits = float(-(hist[hist > 0] * np.log2(p)).sum())
    huff_bits = int(enc["lane_bits"].astype(np.int64).sum())
    freq = quantize(hist)
    lanes = syms.reshape(-1, syms.shape[2])
    rans_lane_bytes = stream_bytes(lanes, nsym.reshape(-1), freq)
    # the same with a separate stream per row (what independent row decoding
    # needs: a second final state per lane)
    if fmt == BF16:
        rows_bits = None
    else:
        half = syms.shape[2] // 2
        rows = np.concatenate([lanes[:, :half], lanes[:, half:]])
        nr = np.full(rows.shape[0], half)
        rows_bits = int(stream_bytes(rows, nr, freq).sum()) * 8
    return dict(symbols=int(hist.sum()), entropy_bits=entropy_bits, huffman_bits=huff_bits,
                rans_bits=int(rans_lane_bytes.sum()) * 8, rans_row_stream_bits=rows_bits,
                lanes=int(lanes.shape[0]))
