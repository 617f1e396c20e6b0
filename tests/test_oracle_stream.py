"""Pins of the oracle's streaming decode (hold back a trailing partial UTF-8
character): the page's worked example, Python's own incremental UTF-8
decoder on every short byte string over the boundary bytes, and round trips."""
import codecs
import itertools
import json
import os

import numpy as np

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "stream_decode.json")


def _table_with(tokens):
    return [bytes([i]) for i in range(256)] + list(tokens)


def test_page_example_hindi_token_boundary():
    g = json.load(open(GOLDEN))
    toks = [bytes.fromhex(h) for h in g["tokens_hex"]]
    table = _table_with(t for t in toks if len(t) > 1)
    enc = oracle.Encoding(table, {})
    ids = [table.index(t) for t in toks]
    dec = oracle.StreamDecoder(enc)
    emits = [dec.feed([i]) for i in ids]
    assert [e.hex() for e in emits] == g["emits_hex"]
    assert dec.finish().hex() == g["final_hex"]


def _python_buffered(b):
    """Bytes Python's incremental UTF-8 decoder keeps for later ('replace' mode
    turns ill-formed bytes into U+FFFD at once; only a possible character
    prefix stays buffered)."""
    d = codecs.getincrementaldecoder("utf-8")("replace")
    d.decode(b, final=False)
    return len(d.getstate()[0])


def test_holdback_matches_python_incremental_decoder():
    alphabet = [0x00, 0x41, 0x7F, 0x80, 0x8F, 0x90, 0x9F, 0xA0, 0xBF, 0xC0, 0xC1, 0xC2, 0xDF,
                0xE0, 0xE1, 0xEC, 0xED, 0xEE, 0xEF, 0xF0, 0xF1, 0xF3, 0xF4, 0xF5, 0xFF]
    n = 0
    for L in range(0, 5):
        for t in itertools.product(alphabet, repeat=L):
            b = bytes(t)
            if len(b) >= 2 and b[-2] == 0xED and 0xA0 <= b[-1] <= 0xBF:
                # the one place Python differs: it buffers the prefix of a
                # surrogate, which no well-formed character completes
                # (Unicode's table of well-formed sequences: after ED comes
                # 80..9F); the oracle emits it
                assert oracle.utf8_holdback(b) == 0 and _python_buffered(b) == 2
                continue
            assert oracle.utf8_holdback(b) == _python_buffered(b), b.hex()
            n += 1
    assert n > 390_000


def test_stream_round_trip_and_valid_chunks(full_table):
    ranks = [(t, i) for i, t in enumerate(full_table)] + workloads.multilingual_table(full_table)
    enc = oracle.Encoding(ranks, {})
    text = workloads.multilingual_text(full_table, n_bytes=60000, seed=9)
    text = text.tobytes() if isinstance(text, np.ndarray) else bytes(text)
    ids = enc.encode(text)
    rng = np.random.default_rng(3)
    for _ in range(5):
        cuts = np.sort(rng.choice(np.arange(1, len(ids)), size=40, replace=False))
        dec = oracle.StreamDecoder(enc)
        out = []
        for a, b in zip(np.r_[0, cuts], np.r_[cuts, len(ids)]):
            e = dec.feed(ids[a:b])
            e.decode("utf-8")  # every emitted chunk is whole characters
            out.append(e)
        out.append(dec.finish())
        assert b"".join(out) == text
