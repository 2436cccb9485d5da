"""The pins also catch mistakes planted in the oracle's C half.

Each case copies ``oracle/lw_oracle.c``, changes one line (a plausible
slip: one package-merge item too few, canonical start codes from the wrong
length count, a comparator that takes the limit itself, bits packed or read
least significant first, a single-precision dot product, decoder bases that
count the length itself), compiles the copy with gcc into a temporary
directory, swaps it in for the oracle's library and re-runs every pin of
``test_oracle_pins.py``: at least one must fail.  Every planted change keeps
the C code inside its buffers (out-of-range indices are still refused by
the decoder's own check), so a mutant can only give wrong answers.  Nothing
here touches liblw or a GPU.  CPU only."""
import os
import shutil
import subprocess

import pytest

import oracle.oracle as O
from test_pin_strength import _failing_pins

SRC = os.path.join(os.path.dirname(O.__file__), "lw_oracle.c")

C_MUTANTS = {
    "package-merge keeps one item too few": (
        "for (int i = 0; i < 2 * n - 2; i++) pm_count",
        "for (int i = 0; i < 2 * n - 3; i++) pm_count"),
    "canonical start codes from the wrong length count": (
        "c = (c + bl_count[b - 1]) << 1;",
        "c = (c + bl_count[b]) << 1;"),
    "comparator takes the limit itself": (
        "if (peek < tb->limit[c]) { L = c; break; }",
        "if (peek <= tb->limit[c]) { L = c; break; }"),
    "codes packed least significant bit first": (
        "for (int i = L - 1; i >= 0; i--) {",
        "for (int i = 0; i < L; i++) {"),
    "lane bits read least significant first": (
        "return (rows[j * 32 + l] >> (31 - (p % 32))) & 1u;",
        "return (rows[j * 32 + l] >> (p % 32)) & 1u;"),
    "dot product accumulated in single precision": (
        "double acc = 0.0;",
        "float acc = 0.0f;"),
    "decoder bases count the length itself": (
        "t->base[L] = b;\n    b += t->count[L];",
        "b += t->count[L];\n    t->base[L] = b;"),
}


def _compile(src_text: str, out_dir) -> str:
    c = os.path.join(out_dir, "lw_oracle.c")
    so = os.path.join(out_dir, "liblw_oracle.so")
    with open(c, "w") as f:
        f.write(src_text)
    subprocess.run(["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-o", so, c], check=True,
                   capture_output=True, text=True)
    return so


def _use(so, monkeypatch):
    """Point the oracle at library `so` for the rest of the test."""
    monkeypatch.setattr(O, "_SO", so)
    monkeypatch.setattr(O, "_lib", None)
    lib = O._load()
    assert lib._name == so


@pytest.fixture(scope="module")
def source():
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    with open(SRC) as f:
        return f.read()


def test_unmutated_copy_passes_every_pin(source, tmp_path, monkeypatch):
    _use(_compile(source, tmp_path), monkeypatch)
    assert _failing_pins() == []


@pytest.mark.parametrize("mutant", sorted(C_MUTANTS))
def test_planted_c_mistake_fails_a_pin(mutant, source, tmp_path, monkeypatch):
    old, new = C_MUTANTS[mutant]
    assert source.count(old) == 1, mutant
    _use(_compile(source.replace(old, new), tmp_path), monkeypatch)
    failed = _failing_pins()
    assert failed, f"no pin catches: {mutant}"
    print(mutant, "->", failed)
