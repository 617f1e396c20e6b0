"""Pins of the oracle's split (the eight clauses of the printed pattern)."""
import itertools
import json
import os

import numpy as np
import pytest

import oracle
from pins import regex_split

HERE = os.path.dirname(os.path.abspath(__file__))


def test_printed_examples():
    """Worked examples printed on the tiktoken page (tests/golden/split_examples.json)."""
    with open(os.path.join(HERE, "golden", "split_examples.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        got = [p.decode() for p in oracle.split(c["text"])]
        assert got == c["pretokens"], (c["text"], got, c["cite"])


# An alphabet that covers every class edge of the pattern: letters (one that
# folds to s), contraction letters, digits (ASCII and Devanagari), space, the
# two CR/LF characters, tab, no-break space, apostrophe, other punctuation, a
# combining mark, an emoji and NUL.
ALPHABET = ["a", "s", "L", "1", " ", "\n", "\r", "\t", "'", ".", "é", "ा", "\U0001F600",
            " ", "\x00", "ſ", "१"]


def _check(s):
    exp = regex_split(s)
    got = oracle.split(s)
    assert got == exp, (s, got, exp)


def test_exhaustive_short_strings():
    """Every string of up to 5 symbols over the 15-symbol alphabet (813,615
    strings), then a seeded sample of 150,000 strings of 6 symbols."""
    pytest.importorskip("regex")
    alpha = ALPHABET[:15]
    n = 0
    for L in range(1, 6):
        for t in itertools.product(alpha, repeat=L):
            _check("".join(t))
            n += 1
    assert n == sum(15 ** k for k in range(1, 6))
    rng = np.random.default_rng(6)
    for row in rng.integers(0, 15, size=(150_000, 6)):
        _check("".join(alpha[i] for i in row))


def test_random_strings():
    pytest.importorskip("regex")
    rng = np.random.default_rng(7)
    for _ in range(20000):
        L = int(rng.integers(1, 65))
        s = "".join(ALPHABET[i] for i in rng.integers(0, len(ALPHABET), size=L))
        _check(s)
    for _ in range(3000):
        L = int(rng.integers(5, 7))
        s = "".join(ALPHABET[i] for i in rng.integers(0, 15, size=L))
        _check(s)


def test_tiling_invariant():
    rng = np.random.default_rng(8)
    for _ in range(2000):
        L = int(rng.integers(0, 40))
        s = "".join(ALPHABET[i] for i in rng.integers(0, len(ALPHABET), size=L))
        b = s.encode()
        parts = oracle.split(b)
        assert b"".join(parts) == b and all(len(p) > 0 for p in parts)


def test_workload_texts_match_library(full_table):
    pytest.importorskip("regex")
    import workloads
    for text in [workloads.tiny_input(), workloads.prose_text(full_table, 256 * 1024, seed=9),
                 workloads.multilingual_text(full_table, 512 * 1024, seed=11)]:
        assert oracle.split(text) == regex_split(text)


# --- the same alternation with r50k's digit clause (" ?\p{N}++") -------------

def test_r50k_digits_printed_examples():
    with open(os.path.join(HERE, "golden", "split_examples_r50k_digits.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        got = [p.decode() for p in oracle.split(c["text"], oracle.PATTERN_R50K_DIGITS)]
        assert got == c["pretokens"], (c["text"], got, c["cite"])


def _check_r50k(s):
    from pins import SPLIT_PATTERN_R50K_DIGITS
    exp = regex_split(s, SPLIT_PATTERN_R50K_DIGITS)
    got = oracle.split(s, oracle.PATTERN_R50K_DIGITS)
    assert got == exp, (s, got, exp)


def test_r50k_digits_exhaustive_short_strings():
    pytest.importorskip("regex")
    alpha = ALPHABET[:15]
    for L in range(1, 5):
        for t in itertools.product(alpha, repeat=L):
            _check_r50k("".join(t))


def test_r50k_digits_random_strings_and_workloads(full_table):
    pytest.importorskip("regex")
    import workloads
    rng = np.random.default_rng(17)
    for _ in range(20000):
        L = int(rng.integers(1, 65))
        _check_r50k("".join(ALPHABET[i] for i in rng.integers(0, len(ALPHABET), size=L)))
    from pins import SPLIT_PATTERN_R50K_DIGITS
    agentic = workloads.pack_segments(workloads.agentic_segments(full_table, seed=3, scale=0.05))[0]
    for text in [agentic, workloads.multilingual_text(full_table, 256 * 1024, seed=12)]:
        text = text.tobytes() if isinstance(text, np.ndarray) else bytes(text)
        assert oracle.split(text, oracle.PATTERN_R50K_DIGITS) == regex_split(text, SPLIT_PATTERN_R50K_DIGITS)
