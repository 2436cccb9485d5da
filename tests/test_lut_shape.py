"""The compact decode table of the table-driven 4-/6-bit product kernel, on the
CPU: its entry count (lw_table_lut_entries, lw_sections.lut_entries) checked
against a brute-force canonical decode of all 2048 peeks.

The kernel indexes its table with max(peek >> s, peek - C).  That is only
correct if every peek mapped to one index decodes to the same codeword, and
the library must pick the smallest such table.  Both are checked here from the
code lengths alone (the oracle's package-merge lengths and hand-made ones),
independently of the library's formula: a codeword's peeks are found by
matching the canonical codes bit by bit, and every s and every offset is tried.
No GPU."""
import numpy as np
import pytest

import oracle
from decode_gemv_gb300 import inputs
from decode_gemv_gb300 import lw


@pytest.fixture(scope="module", autouse=True)
def built():
    lw.load()


def peek_codewords(code_len):
    """For every 11-bit peek, the (symbol, length) of the canonical codeword
    it starts with (brute force: the code that is a prefix of the peek)."""
    code_len = np.asarray(code_len, dtype=np.int64)
    codes = oracle.canonical_codes(code_len)
    out = np.full((2048, 2), -1, np.int64)
    for p in range(2048):
        for s, L in enumerate(code_len):
            if L and (p >> (11 - L)) == codes[s]:
                out[p] = (s, L)
                break
    return out


def smallest_consistent_table(cw):
    """Smallest n over (s, C) such that index(p) = max(p >> s, p - C) gives
    every index one codeword and the indices are exactly 0..n-1."""
    best = 2048
    peeks = np.arange(2048)
    for s in range(1, 11):
        for C in range(0, 2048):
            idx = np.maximum(peeks >> s, peeks - C)
            n = int(idx.max()) + 1
            if n >= best or len(np.unique(idx)) != n:
                continue
            first = np.full((n, 2), -1, np.int64)
            first[idx[::-1]] = cw[::-1]
            if np.array_equal(first[idx], cw):
                best = n
    return best


def table_of(code_len, fmt):
    return lw.lw_table_from_lengths(fmt, np.asarray(code_len, np.uint8))


@pytest.mark.parametrize("sd", [1.2, 1.6, 2.2])
def test_lut_entries_of_workload_tables_are_minimal_and_consistent(sd):
    m = inputs.small_q4(3, 256, 2048, sd=sd)
    counts = np.bincount(oracle.q4_pair_symbols(m["codes"]).ravel(), minlength=256)
    L = oracle.code_lengths(counts)
    n = lw.lw_table_lut_entries(table_of(L, lw.LW_FMT_Q4_PAIR))
    assert 1 <= n <= 512            # the workloads' tables fit the kernel
    assert n == smallest_consistent_table(peek_codewords(L))


def test_lut_entries_of_a_six_bit_table():
    m = inputs.small_q6(4, 128, 1024)
    L = oracle.code_lengths(np.bincount(m["codes"].ravel(), minlength=64))
    n = lw.lw_table_lut_entries(table_of(L, lw.LW_FMT_Q6))
    assert n == smallest_consistent_table(peek_codewords(L))


def test_lut_entries_special_tables():
    # a lone symbol (length 1, the table completes it with a phantom code)
    L = np.zeros(256, np.uint8)
    L[7] = 1
    assert lw.lw_table_lut_entries(table_of(L, lw.LW_FMT_Q4_PAIR)) == 2
    # 256 symbols of length 8: every 8-bit prefix is a codeword
    assert lw.lw_table_lut_entries(table_of(np.full(256, 8), lw.LW_FMT_Q4_PAIR)) == 256
    # a skewed table: one symbol of length 1 and long codes filling the rest
    # (67 of length 8, 100 of length 9, 88 of length 11; Kraft sum in units
    # of 2^-11: 1024 + 536 + 400 + 88 = 2048): every compaction leaves more
    # than the kernel's 512 entries, so the library routes such a matrix to
    # the comparator kernel
    L = np.zeros(256, np.int64)
    L[0] = 1
    L[1:68] = 8
    L[68:168] = 9
    L[168:256] = 11
    assert int(sum(2 ** (11 - int(v)) for v in L if v)) == 2048
    n = lw.lw_table_lut_entries(table_of(L, lw.LW_FMT_Q4_PAIR))
    assert n == 578 > 512
    assert n == smallest_consistent_table(peek_codewords(L))


def test_bundle_stats_carry_the_hint():
    m = inputs.small_q4(5, 128, 512)
    hb = lw.lw_encode_bundle(lw.LW_FMT_Q4_PAIR, m["codes"], m["scales"], m["mins"])
    assert hb.stats.lut_entries == lw.lw_table_lut_entries(hb.sections["table"])
    tw = lw.lw_encode_bundle(lw.LW_FMT_Q4_PAIR, m["codes"], m["scales"], m["mins"], twin=True)
    assert tw.stats.lut_entries == 0
    b = inputs.small_bf16(6, 64, 512)
    hbb = lw.lw_encode_bundle(lw.LW_FMT_BF16_EXP, b["bits"])
    n = lw.lw_table_lut_entries(hbb.sections["table"])
    assert hbb.stats.lut_entries == n and 1 <= n <= 512
    bt = lw.lw_encode_bundle(lw.LW_FMT_BF16_EXP, b["bits"], twin=True)
    assert bt.stats.lut_entries == 0


def test_workload_bf16_tables_fit():
    """The Llama MLP's exponent tables (16-symbol palettes): their compact
    tables are those of brute force and fit the kernel's 512 entries."""
    spec = inputs.workload_specs(inputs.LLAMA_MLP_BF16)[0]
    rng = inputs.matrix_rng(inputs.LLAMA_MLP_BF16, 0, 0)
    w = inputs.bf16_matrix(rng, 256, spec.cols)["bits"]
    hb = lw.lw_encode_bundle(lw.LW_FMT_BF16_EXP, w)
    L = lw.table_fields(hb.sections["table"])["code_len"][:16]
    n = hb.stats.lut_entries
    assert n == smallest_consistent_table(peek_codewords(L)) and 1 <= n <= 512


def test_device_view_computes_the_hint_when_not_given():
    """A device view built from host sections without the bundle's stats (as
    a bundle rebuilt in another process is) still carries the compact-table
    size, so its products take the table-driven kernel (views on the CPU)."""
    pytest.importorskip("torch")
    m = inputs.small_q4(11, 256, 1024)
    hb = lw.lw_encode_bundle(lw.LW_FMT_Q4_PAIR, m["codes"], m["scales"], m["mins"])
    args = (hb.desc.fmt, hb.desc.twin, hb.desc.rows, hb.desc.cols, hb.sections,
            hb.stats.max_tile_rows, hb.stats.min_len, hb.stats.max_len)
    db = lw.DeviceBundle(*args, device="cpu")
    assert hb.stats.lut_entries > 0 and db.view.lut_entries == hb.stats.lut_entries
    tw = lw.lw_encode_bundle(lw.LW_FMT_Q4_PAIR, m["codes"], m["scales"], m["mins"], twin=True)
    dt = lw.DeviceBundle(tw.desc.fmt, tw.desc.twin, tw.desc.rows, tw.desc.cols, tw.sections,
                         tw.stats.max_tile_rows, tw.stats.min_len, tw.stats.max_len, device="cpu")
    assert dt.view.lut_entries == 0
