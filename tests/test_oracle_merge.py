"""Pins of the oracle's merge loop: brute force on tiny inputs, closed forms."""
import itertools

import numpy as np
import pytest

import oracle
from pins import naive_bpe


def _random_table(rng, alphabet, n_tok, tie_free=True):
    """Byte floor + random concatenations of existing tokens over `alphabet`."""
    toks = [bytes([b]) for b in range(256)]
    have = set(toks)
    base = [bytes([c]) for c in alphabet]
    pool = list(base)
    tries = 0
    while len(toks) < 256 + n_tok and tries < 10000:
        tries += 1
        t = pool[int(rng.integers(0, len(pool)))] + pool[int(rng.integers(0, len(pool)))]
        if len(t) > 6 or t in have:
            continue
        have.add(t)
        toks.append(t)
        pool.append(t)
    # shuffle the ranks of the merged tokens (keeps them unique: no ties by construction
    # of distinct ids, but adjacent equal pairs such as "aa" give leftmost-tie cases)
    merged = toks[256:]
    perm = rng.permutation(len(merged))
    return toks[:256] + [merged[i] for i in perm]


@pytest.mark.parametrize("alphabet,maxlen", [(b"ab", 10), (b"abc", 8), (b"abcd", 8)])
def test_exhaustive_against_brute_force(alphabet, maxlen):
    """Every string of up to maxlen symbols, on 20 seeded random tables per
    alphabet (repeated symbols give the equal-rank pairs where the leftmost
    tie-break decides)."""
    rng = np.random.default_rng(len(alphabet))
    n_tables = 20
    for t in range(n_tables):
        table = _random_table(rng, alphabet, int(rng.integers(3, 40)))
        ranks = {tok: i for i, tok in enumerate(table)}
        enc = oracle.Encoding(table)
        for L in range(1, maxlen + 1):
            for s in itertools.product(alphabet, repeat=L):
                piece = bytes(s)
                got = list(enc.bpe_piece(piece))
                assert got == naive_bpe(piece, ranks), (table[256:], piece)


def test_random_full_bytes_against_brute_force():
    rng = np.random.default_rng(99)
    for t in range(10):
        alphabet = bytes(rng.choice(256, size=6, replace=False).astype(np.uint8))
        table = _random_table(rng, alphabet, 60)
        ranks = {tok: i for i, tok in enumerate(table)}
        enc = oracle.Encoding(table)
        for _ in range(500):
            piece = bytes(rng.choice(list(alphabet), size=int(rng.integers(1, 9))).astype(np.uint8))
            assert list(enc.bpe_piece(piece)) == naive_bpe(piece, ranks)


def test_closed_forms():
    byte_only = [bytes([b]) for b in range(256)]
    enc = oracle.Encoding(byte_only)
    s = bytes(range(128)) * 2 + "é中😀".encode()
    assert list(enc.encode(s)) == list(s)  # bytes-only table: ids are the bytes
    for b in range(256):
        assert list(enc.bpe_piece(bytes([b]))) == [b]
    enc = oracle.Encoding(byte_only + [b"aa"])
    assert list(enc.bpe_piece(b"aaaa")) == [256, 256]
    assert list(enc.bpe_piece(b"aaa")) == [256, ord("a")]  # leftmost tie-break
    assert list(enc.bpe_piece(b"a")) == [ord("a")]


def test_final_pairs_are_not_tokens(full_enc, full_table):
    """At the end of the loop no adjacent pair of output tokens concatenates to
    a token (the loop stops only when every pair rank is MAX)."""
    import workloads
    have = set(full_table)
    text = workloads.prose_text(full_table, 64 * 1024, seed=21)
    for piece in oracle.split(text)[:3000]:
        ids = list(full_enc.bpe_piece(piece))
        toks = [full_table[i] for i in ids]
        assert b"".join(toks) == piece
        for a, b in zip(toks, toks[1:]):
            assert a + b not in have


def test_table_validation():
    floor = [bytes([b]) for b in range(256)]
    with pytest.raises(oracle.OracleError):
        oracle.Encoding(floor[:255])  # a missing byte breaks the byte floor
    with pytest.raises(oracle.OracleError):
        oracle.Encoding(floor + [b"ab", b"ab"])  # duplicate bytes
    with pytest.raises(oracle.OracleError):
        oracle.Encoding(floor, {"<|x|>": 65})  # special id collides with a rank


def test_token_unreachable_from_its_own_bytes():
    """Worked by hand: ranks bc=256 < ab=257 < cd=258 < abcd=259.  The loop
    merges the least rank first (bc), after which no pair of [a, bc, d] is a
    token, so "abcd" never becomes the token abcd."""
    table = [bytes([i]) for i in range(256)] + [b"bc", b"ab", b"cd", b"abcd"]
    enc = oracle.Encoding(table, {})
    assert list(enc.bpe_piece(b"abcd")) == [ord("a"), 256, ord("d")]
    assert list(enc.bpe_piece(b"abcdab")) == [ord("a"), 256, ord("d"), 257]
