"""Pins of the tiktoken-safe chunking (400k-character windows, 25k runs)."""
import numpy as np

import oracle
from pins import closed_form_cuts


def _oracle_cut_chars(text):
    chunks = oracle.safe_chunks(text)
    cuts, pos = [], 0
    for c in chunks:
        cuts.append(pos)
        pos += len(c.decode())
    return cuts


def test_py_isspace_matches_python():
    for c in range(0x110000):
        if 0xD800 <= c <= 0xDFFF:
            continue
        assert oracle.py_isspace(c) == chr(c).isspace(), hex(c)


def test_60k_space_run():
    text = "ab" + " " * 60000 + "cd"
    assert _oracle_cut_chars(text) == [0, 2 + 25000, 2 + 50000]


def test_window_cut_with_multibyte_neighbours():
    text = "é" * 399_999 + "中" + "🙂" * 5 + "x" * 10
    cuts = _oracle_cut_chars(text)
    # the non-space run is cut every 25,000 characters; the window restarts at 400,000
    assert 400_000 in cuts
    assert cuts == closed_form_cuts([ch.isspace() for ch in text])


def test_random_run_structures_match_closed_form():
    rng = np.random.default_rng(5)
    for _ in range(30):
        parts = []
        n = 0
        while n < int(rng.integers(10_000, 900_000)):
            L = int(np.exp(rng.uniform(0, np.log(80_000))))
            ch = [" ", "\n", "\t", "a", "é", "中", "\x1c"][int(rng.integers(0, 7))]
            parts.append(ch * L)
            n += L
        text = "".join(parts)
        assert _oracle_cut_chars(text) == closed_form_cuts([c.isspace() for c in text])


def test_empty_and_single():
    assert oracle.safe_chunks(b"") == []
    assert oracle.safe_chunks(b"x") == [b"x"]
