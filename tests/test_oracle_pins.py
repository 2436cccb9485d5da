"""Pins for the CPU oracle: checks against brute force, exhaustive search,
closed forms, a textbook Huffman, an RFC worked example and invariants -- never
against the oracle itself.  CPU only."""
import heapq
import itertools
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from decode_gemv_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- helpers

def textbook_huffman_lengths(counts):
    """Unrestricted Huffman with a heap (merging the two lightest trees)."""
    items = [(c, i, [s]) for i, (s, c) in enumerate((s, c) for s, c in enumerate(counts) if c)]
    if len(items) == 1:
        return {items[0][2][0]: 1}
    heapq.heapify(items)
    depth = {s: 0 for _, _, ss in items for s in ss}
    uid = len(items)
    while len(items) > 1:
        c1, _, s1 = heapq.heappop(items)
        c2, _, s2 = heapq.heappop(items)
        for s in s1 + s2:
            depth[s] += 1
        heapq.heappush(items, (c1 + c2, uid, s1 + s2))
        uid += 1
    return depth


def cost(counts, lengths):
    return sum(int(c) * int(l) for c, l in zip(counts, lengths))


def kraft(lengths):
    return sum(Fraction(1, 2 ** int(l)) for l in lengths if l)


def bitstr(code, length):
    return format(int(code), f"0{int(length)}b")


def q4_pair_hist(sd, seed=0, shape=(256, 4096)):
    rng = np.random.default_rng(seed)
    c = np.clip(np.rint(rng.normal(7.5, sd, size=shape)), 0, 15).astype(np.uint8)
    return np.bincount(oracle.q4_pair_symbols(c).ravel(), minlength=256)


# ---------------------------------------------------------------- lengths

def test_package_merge_matches_exhaustive_search():
    """Optimality under the length limit: exhaustive search over all length
    vectors that satisfy Kraft and the limit gives the same minimum cost."""
    rng = np.random.default_rng(123)
    for trial in range(60):
        n = int(rng.integers(2, 7))
        lmax = int(rng.integers(max(1, math.ceil(math.log2(n))), 5))
        counts = [int(v) for v in rng.integers(1, 50, size=n)]
        if trial % 3 == 0:               # skewed, so the limit binds
            counts = [int(2 ** (i * 2) + v) for i, v in enumerate(counts)]
        best = None
        for ls in itertools.product(range(1, lmax + 1), repeat=n):
            if kraft(ls) <= 1:
                c = cost(counts, ls)
                best = c if best is None else min(best, c)
        got = oracle.code_lengths(counts, lmax)
        assert max(got) <= lmax
        assert kraft(got) <= 1
        assert cost(counts, got) == best, (counts, lmax, got)


def test_equals_textbook_huffman_when_limit_does_not_bind():
    rng = np.random.default_rng(7)
    checked = 0
    for _ in range(40):
        n = int(rng.integers(2, 64))
        counts = rng.integers(1, 1000, size=n).tolist()
        tb = textbook_huffman_lengths(counts)
        if max(tb.values()) > 11:
            continue
        got = oracle.code_lengths(counts, 11)
        assert cost(counts, got) == sum(counts[s] * l for s, l in tb.items())
        checked += 1
    assert checked > 20


@pytest.mark.parametrize("sd", [1.2, 1.6, 2.2])
def test_q4_pair_tables_are_complete_and_limited(sd):
    h = q4_pair_hist(sd)
    got = oracle.code_lengths(h, 11)
    used = h > 0
    assert (got[used] >= 1).all() and (got[~used] == 0).all()
    assert got.max() <= 11
    assert kraft(got) == 1                      # complete code
    tb = textbook_huffman_lengths(h.tolist())
    unlimited = sum(int(h[s]) * l for s, l in tb.items())
    assert max(tb.values()) > 11                # the 11-bit limit binds here
    assert cost(h, got) >= unlimited
    # entropy bound per symbol: H <= mean length < H + 1 (+ small limit loss)
    p = h[used] / h.sum()
    H = float(-(p * np.log2(p)).sum())
    mean = cost(h, got) / h.sum()
    assert H <= mean < H + 1
    assert mean - cost(h, [tb.get(s, 0) for s in range(256)]) / h.sum() < 0.1


def test_q4_sd16_rate_matches_estimate():
    """Rate sanity for the tiny workload's distribution: about 2.75 bits of
    entropy per 4-bit code, and the coded rate lands just above it."""
    h = q4_pair_hist(1.6)
    got = oracle.code_lengths(h, 11)
    per_code = cost(h, got) / h.sum() / 2
    assert 2.74 < per_code < 2.82


def test_edge_lengths():
    assert list(oracle.code_lengths([0, 9, 0])) == [0, 1, 0]
    assert list(oracle.code_lengths([0, 0, 0])) == [0, 0, 0]
    assert list(oracle.code_lengths([3, 3])) == [1, 1]
    uni = oracle.code_lengths([5] * 256)
    assert (uni == 8).all()
    # all 2048 codes of length 11 when 2048 symbols are equally likely
    assert (oracle.code_lengths([1] * 2048, 11) == 11).all()
    with pytest.raises(ValueError):
        oracle.code_lengths([1] * 2049, 11)


# ---------------------------------------------------------------- canonical

def test_canonical_rfc1951_worked_example():
    rows = [l.split() for l in open(os.path.join(GOLDEN, "rfc1951_canonical.txt"))
            if l.strip() and not l.startswith("#")]
    lengths = [int(r[1]) for r in rows]
    codes = oracle.canonical_codes(lengths)
    for (_, L, want), got in zip(rows, codes):
        assert bitstr(got, L) == want


def test_canonical_codes_are_prefix_free_and_ordered():
    rng = np.random.default_rng(5)
    for sd in (1.2, 2.2):
        h = q4_pair_hist(sd, seed=int(rng.integers(1000)), shape=(64, 1024))
        L = oracle.code_lengths(h, 11)
        C = oracle.canonical_codes(L)
        strs = {s: bitstr(C[s], L[s]) for s in range(256) if L[s]}
        items = list(strs.items())
        for (a, sa), (b, sb) in itertools.combinations(items, 2):
            assert not sa.startswith(sb) and not sb.startswith(sa)
        # canonical: ordered by (length, symbol) the codes are increasing when
        # left-aligned, and consecutive within one length
        order = sorted(strs, key=lambda s: (L[s], s))
        vals = [int(strs[s].ljust(11, "0"), 2) for s in order]
        assert vals == sorted(vals) and len(set(vals)) == len(vals)
        for s1, s2 in zip(order, order[1:]):
            if L[s1] == L[s2]:
                assert C[s2] == C[s1] + 1


def test_decoder_tables_against_brute_force_peeks():
    """For every 11-bit peek, the comparator quantities select the codeword
    found by searching all codes for the one that prefixes the peek."""
    h = q4_pair_hist(1.6, shape=(64, 2048))
    L = oracle.code_lengths(h, 11)
    C = oracle.canonical_codes(L)
    t = oracle.decoder_tables(L)
    for peek in range(2048):
        p = format(peek, "011b")
        hits = [s for s in range(256) if L[s] and p.startswith(bitstr(C[s], L[s]))]
        assert len(hits) == 1
        s = hits[0]
        # the limit of length L[s] is the first one above the peek
        cand = [l for l in range(1, 12) if peek < int(t["limit"][l])]
        assert cand[0] == L[s]
        ls = int(L[s])
        idx = int(t["base"][ls]) + (peek >> (11 - ls)) - int(t["first_code"][ls])
        assert t["sorted"][idx] == s


# ---------------------------------------------------------------- lanes

def expected_lane_bits(lane_syms, L, C):
    return "".join(bitstr(C[s], L[s]) for s in lane_syms)


def test_lane_layout_brute_force_q4():
    m = inputs.small_q4(11, 128, 512)
    b = oracle.encode(oracle.Q4, m["codes"])
    L, C = b["code_len"], oracle.canonical_codes(b["code_len"])
    codes = m["codes"]
    tk = 512 // 256
    for t in range((128 // 64) * tk):
        s, kt = divmod(t, tk)
        strs = []
        for l in range(32):
            syms = []
            for r in (64 * s + 2 * l, 64 * s + 2 * l + 1):
                for k in range(256 * kt, 256 * kt + 256, 2):
                    syms.append(int(codes[r, k]) | int(codes[r, k + 1]) << 4)
            strs.append(expected_lane_bits(syms, L, C))
        wt = max((len(x) + 31) // 32 for x in strs)
        assert b["tile_off"][t + 1] - b["tile_off"][t] == wt
        for l, x in enumerate(strs):
            assert b["lane_bits"][t, l] == len(x)
            first_row = [int(codes[64 * s + 2 * l, k]) | int(codes[64 * s + 2 * l, k + 1]) << 4
                         for k in range(256 * kt, 256 * kt + 256, 2)]
            assert b["lane_mid"][t, l] == len(expected_lane_bits(first_row, L, C))
            x = x.ljust(32 * wt, "0")
            for j in range(wt):
                word = b["words"][(b["tile_off"][t] + j) * 32 + l]
                assert format(int(word), "032b") == x[32 * j: 32 * j + 32]


@pytest.mark.parametrize("fmt,maker", [(oracle.Q4, lambda: inputs.small_q4(3, 192, 768)),
                                       (oracle.Q6, lambda: inputs.small_q6(4, 128, 512))])
def test_roundtrip_and_textbook_decode(fmt, maker):
    m = maker()
    b = oracle.encode(fmt, m["codes"])
    out = oracle.decode(fmt, m["codes"].shape[0], m["codes"].shape[1],
                        b["code_len"], b["words"], b["tile_off"])
    if fmt == oracle.Q4:
        assert np.array_equal(oracle.unpack_q4(out), m["codes"])
    else:
        assert np.array_equal(out, m["codes"])
    # one lane decoded bit by bit against the code book
    L, C = b["code_len"], oracle.canonical_codes(b["code_len"])
    book = {bitstr(C[s], L[s]): s for s in range(len(L)) if L[s]}
    t, l = 1, 17
    wt = b["tile_off"][t + 1] - b["tile_off"][t]
    stream = "".join(format(int(b["words"][(b["tile_off"][t] + j) * 32 + l]), "032b")
                     for j in range(wt))
    syms, cur = [], ""
    for bit in stream[: b["lane_bits"][t, l]]:
        cur += bit
        if cur in book:
            syms.append(book[cur])
            cur = ""
    assert cur == ""
    dec, used = oracle.decode_lanes(b["code_len"], b["words"], b["tile_off"], b["nsym"],
                                    256 if fmt == oracle.Q4 else 512)
    assert list(dec[t, l]) == syms
    assert np.array_equal(used, b["lane_bits"].astype(np.uint32))


def test_roundtrip_edge_cases():
    # a single symbol everywhere: length-1 code, 8 words per lane
    z = np.full((64, 256), 9, dtype=np.uint8)
    b = oracle.encode(oracle.Q4, z)
    assert (b["code_len"] > 0).sum() == 1 and b["tile_off"][-1] == 8
    assert np.array_equal(oracle.unpack_q4(oracle.decode(oracle.Q4, 64, 256, b["code_len"], b["words"], b["tile_off"])), z)
    # one lane far longer than the rest: rare symbols in rows 0 and 1 only
    rng = np.random.default_rng(0)
    c = np.full((64, 512), 7, dtype=np.uint8)
    c[:2, :256] = rng.integers(0, 16, size=(2, 256))
    b = oracle.encode(oracle.Q4, c)
    lb = b["lane_bits"]
    assert lb[0, 0] > 4 * lb[0, 1]
    assert np.array_equal(oracle.unpack_q4(oracle.decode(oracle.Q4, 64, 512, b["code_len"], b["words"], b["tile_off"])), c)
    # many maximum-length codes: a near-uniform tail under a dominant symbol
    c = np.full((64, 256), 0, dtype=np.uint8)
    c[:, 1::2] = rng.integers(0, 16, size=(64, 128))
    c[::2, ::4] = rng.integers(0, 16, size=(32, 64))
    b = oracle.encode(oracle.Q4, c)
    assert b["code_len"].max() <= 11
    assert np.array_equal(oracle.unpack_q4(oracle.decode(oracle.Q4, 64, 256, b["code_len"], b["words"], b["tile_off"])), c)


# ---------------------------------------------------------------- BF16

def test_bf16_split_join_exhaustive():
    allb = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    e, s = oracle.bf16_fields(allb)
    assert np.array_equal(oracle.bf16_join(e, s), allb)
    # field meaning: value = (-1)^sign * 2^(e-127) * (1 + mantissa/128), normal range
    v = oracle.bf16_to_f64(allb)
    normal = (e > 0) & (e < 255)
    mant = (s & 0x7F).astype(np.float64)
    sign = np.where(s & 0x80, -1.0, 1.0)
    want = sign * np.ldexp(1.0 + mant / 128.0, e.astype(np.int64) - 127)
    assert np.array_equal(v[normal], want[normal])


def test_bf16_to_f64_matches_torch():
    torch = pytest.importorskip("torch")
    bits = np.random.default_rng(1).integers(0, 65536, size=4096).astype(np.uint16)
    t = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy().astype(np.float64)
    ours = oracle.bf16_to_f64(bits)
    fin = np.isfinite(t)
    assert np.array_equal(ours[fin], t[fin])


def test_palette_and_verbatim_rule_brute_force():
    m = inputs.small_bf16(5, 128, 512, outlier_p=0.01)
    sp = oracle.bf16_split(m["bits"])
    exp = sp["exp"]
    counts = {}
    for e in exp.ravel().tolist():
        counts[e] = counts.get(e, 0) + 1
    top = sorted(sorted(counts, key=lambda e: (-counts[e], e))[:16])
    assert list(sp["palette"]) == top
    pal = set(top)
    n, k = exp.shape
    for r in range(n):
        for g in range(k // 64):
            outside = [e for e in exp[r, 64 * g: 64 * g + 64].tolist() if e not in pal]
            assert sp["verbatim"][r, g] == (len(outside) > 0)
    assert 0 < sp["verbatim"].mean() < 1


@pytest.mark.parametrize("p", [0.0, 0.002, 1.0])
def test_bf16_roundtrip(p):
    m = inputs.small_bf16(6, 128, 512, outlier_p=p)
    bits = m["bits"]
    if p == 1.0:
        # every group verbatim: 16 common exponents everywhere, and column 0 of
        # each group takes one of 40 rare exponents (each far less frequent)
        r, k = np.indices(bits.shape)
        exp = (100 + (r * 7 + k) % 16).astype(np.uint16)
        exp[:, ::64] = 200 + (r[:, ::64] * 8 + k[:, ::64] // 64) % 40
        bits = (bits & 0x807F) | (exp << 7)
    b = oracle.encode(oracle.BF16, bits)
    if p == 1.0:
        assert b["verbatim"].all()
    if p == 0.0:
        assert b["verbatim"].mean() < 0.01
    out = oracle.decode(oracle.BF16, 128, 512, b["code_len"], b["words"], b["tile_off"],
                        palette=b["palette"], verbatim=b["verbatim"], vexp=b["vexp"], sm=b["sm"])
    assert np.array_equal(out, bits)


def test_bf16_workload_statistics():
    """The BF16 workload's exponents: the top-16 palette covers over 99 % of
    weights and the palette-index entropy is near 2.6 bits (Unweight, "The
    exponent's exploitable redundancy")."""
    m = inputs.small_bf16(7, 512, 4096)
    sp = oracle.bf16_split(m["bits"])
    inpal = np.isin(sp["exp"], sp["palette"]).mean()
    assert inpal > 0.99
    idx = sp["index"][sp["index"] != 255]
    p = np.bincount(idx, minlength=16) / idx.size
    p = p[p > 0]
    H = float(-(p * np.log2(p)).sum())
    assert 2.3 < H < 2.9


# ---------------------------------------------------------------- arithmetic

def test_gemm_against_exact_sums():
    rng = np.random.default_rng(9)
    w = rng.standard_normal((5, 300))
    x = rng.standard_normal((2, 300))
    y = oracle.gemm(w, x)
    for b in range(2):
        for r in range(5):
            exact = math.fsum(float(a) * float(c) for a, c in zip(w[r], x[b]))
            assert abs(y[b, r] - exact) <= 1e-13 * sum(abs(w[r] * x[b]))


def test_q4_gemv_closed_forms():
    m = inputs.small_q4(2, 64, 512)
    codes, sc, mn = m["codes"], m["scales"], m["mins"]
    s = oracle.fp16_to_f64(sc)
    mi = oracle.fp16_to_f64(mn)
    W = oracle.dequant_q4(codes, sc, mn)
    # one-hot x picks a dequantised column
    for k in (0, 255, 256, 511):
        x = np.zeros((1, 512))
        x[0, k] = 1.0
        assert np.array_equal(oracle.gemm(W, x)[0], s[:, k // 256] * codes[:, k] + mi[:, k // 256])
    # constant codes: y_r = sum_b (s_b c + m_b) * sum_{k in b} x_k
    x = m["x"].astype(np.float64)
    cc = np.full_like(codes, 5)
    y = oracle.gemm(oracle.dequant_q4(cc, sc, mn), x)[0]
    xb = x[0].reshape(2, 256).sum(axis=1)
    want = ((s * 5 + mi) * xb).sum(axis=1)
    assert np.allclose(y, want, rtol=1e-12, atol=1e-12)
    # x = 1: row sums; zero codes and zero mins: exactly zero
    assert np.allclose(oracle.gemm(W, np.ones((1, 512)))[0], W.sum(axis=1), rtol=1e-13)
    z = oracle.dequant_q4(np.zeros_like(codes), sc, np.zeros_like(mn))
    assert (oracle.gemm(z, x) == 0).all()


def test_q4_lattice_idempotence():
    """Re-quantising a dequantised weight gives back its code exactly
    (Software-Defined Bandwidth, section IV.A: the codec is idempotent on its
    lattice)."""
    m = inputs.small_q4(8, 128, 512)
    W = oracle.dequant_q4(m["codes"], m["scales"], m["mins"])
    s = np.repeat(oracle.fp16_to_f64(m["scales"]), 256, axis=1)
    mi = np.repeat(oracle.fp16_to_f64(m["mins"]), 256, axis=1)
    assert np.array_equal(np.rint((W - mi) / s).astype(np.uint8), m["codes"])


def test_q6_dequant_closed_form():
    m = inputs.small_q6(3, 64, 256)
    W = oracle.dequant_q6(m["codes"], m["scales"])
    r, k = 10, 37
    want = float(np.float16(m["scales"].view(np.float16)[r, k // 16])) * (int(m["codes"][r, k]) - 32)
    assert W[r, k] == want
    c32 = np.full_like(m["codes"], 32)
    assert (oracle.dequant_q6(c32, m["scales"]) == 0).all()


def test_twin_layout_brute_force():
    m = inputs.small_q4(12, 64, 256)
    w = oracle.twin_words(oracle.Q4, m["codes"])
    assert w.size == 64 * 32
    c = m["codes"]
    for l in (0, 5, 31):
        stream = "".join(format(int(v), "04b") for r in (2 * l, 2 * l + 1) for v in c[r])
        for j in (0, 31, 63):
            assert format(int(w[j * 32 + l]), "032b") == stream[32 * j: 32 * j + 32]
    m6 = inputs.small_q6(12, 64, 256)
    w6 = oracle.twin_words(oracle.Q6, m6["codes"])
    assert w6.size == 96 * 32
    stream = "".join(format(int(v), "06b") for r in (2, 3) for v in m6["codes"][r])
    assert format(int(w6[7 * 32 + 1]), "032b") == stream[224:256]


def test_bf16_twin_layout_brute_force():
    """The BF16 twin: every weight's exponent as a 4-bit index into the
    ascending top-16 palette, 0 throughout a verbatim 64-column group; the
    palette and the verbatim groups counted here by hand."""
    m = inputs.small_bf16(13, 64, 512, outlier_p=0.01)
    bits = m["bits"]
    exp = [[(int(v) >> 7) & 0xFF for v in row] for row in bits]
    counts = {}
    for row in exp:
        for e in row:
            counts[e] = counts.get(e, 0) + 1
    palette = sorted(sorted(counts, key=lambda e: (-counts[e], e))[:16])
    assert len(counts) > 16                       # some groups are verbatim
    pos = {e: i for i, e in enumerate(palette)}
    w = oracle.twin_words(oracle.BF16, bits)
    assert w.size == 2 * 64 * 32                  # 2 tiles, 64 words per lane
    n_verbatim = 0
    for t in range(2):
        for l in (0, 9, 31):
            vals = []
            for r in (2 * l, 2 * l + 1):
                for g in range(4 * t, 4 * t + 4):
                    grp = exp[r][64 * g: 64 * g + 64]
                    if all(e in pos for e in grp):
                        vals += [pos[e] for e in grp]
                    else:
                        vals += [0] * 64
                        n_verbatim += 1
            stream = "".join(format(v, "04b") for v in vals)
            for j in range(64):
                assert format(int(w[t * 64 * 32 + j * 32 + l]), "032b") == stream[32 * j: 32 * j + 32]
    assert n_verbatim > 0
