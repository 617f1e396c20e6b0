"""End-to-end invariants of the oracle on the workloads."""
import numpy as np
import pytest

import oracle
import workloads


def test_byte_floor(full_table):
    assert all(bytes([b]) in set(full_table) for b in range(256))
    assert full_table[:256] == [bytes([b]) for b in range(256)]


def test_round_trip_special_strings(full_enc):
    s = "NUL:\x00 emoji:\U0001F600 CJK:中文 replaced:� end".encode()
    assert full_enc.decode(full_enc.encode(s)) == s


def test_invalid_utf8_rejected(full_enc):
    for bad in [b"\xff", b"a\xc0\x80", b"\xed\xa0\x80", b"\xe4\xb8", b"\x80"]:
        with pytest.raises(oracle.OracleError):
            full_enc.encode(bad)


def test_pretoken_ids_decode_to_pretoken(full_enc, full_table):
    text = workloads.prose_text(full_table, 32 * 1024, seed=31)
    for p in oracle.split(text):
        assert full_enc.decode(full_enc.bpe_piece(p)) == p


def test_specials_policy(full_enc):
    sp = workloads.SPECIALS
    only = "".join(sp)
    ids, off = full_enc.encode_segments([(only, True)])
    assert list(ids) == list(sp.values())
    ids_f, _ = full_enc.encode_segments([(only, False)])
    assert not set(ids_f) & set(sp.values())
    assert full_enc.decode(ids_f) == only.encode()
    ids, off = full_enc.encode_segments([("x<|endoftext|>y", True), ("x<|endoftext|>y", False),
                                         ("", True), ("z", False)])
    assert list(off) == [0, 3, 3 + len(ids) - 4, len(ids) - 1, len(ids)] or off[-1] == len(ids)
    assert ids[1] == 100257
    assert 100257 not in list(ids[off[1]:off[2]])
    assert off[2] == off[3]


def test_special_cut_by_chunk_boundary_is_ordinary(full_enc):
    # a special straddling a 25k-run cut (non-space run of 25,000+ characters)
    text = "x" * 24_995 + "<|endoftext|>"
    ids, _ = full_enc.encode_segments([(text, True)], tiktoken_safe=True)
    assert 100257 not in list(ids)
    ids, _ = full_enc.encode_segments([(text, True)], tiktoken_safe=False)
    assert 100257 in list(ids)


def test_workloads_round_trip(full_enc, full_table, tiny_enc):
    text = workloads.tiny_input()
    assert tiny_enc.decode(tiny_enc.encode(text)) == text
    text = workloads.prose_text(full_table, 256 * 1024, seed=2)
    assert full_enc.decode(full_enc.encode(text)) == text
    segs = workloads.agentic_segments(full_table, seed=3, scale=0.02)
    ids, off = full_enc.encode_segments(segs, tiktoken_safe=True)
    assert full_enc.decode(ids) == b"".join(s for s, _ in segs)
    for k, (s, allow) in enumerate(segs):
        if not allow:
            assert not set(ids[off[k]:off[k + 1]].tolist()) & set(workloads.SPECIALS.values())


def test_tiny_table_shape(tiny_table):
    assert len(tiny_table) == 256 + 4096
    have = set(tiny_table[:256])
    for t in tiny_table[256:]:
        assert any(t[:k] in have and t[k:] in have for k in range(1, len(t)))
        have.add(t)


def test_trainer_matches_brute_force():
    """The plain trainer that builds the tiny table, against a brute-force
    trainer (tests/pins.py) that recounts pairs from the regex library's split:
    a slice of the tiny corpus and tie-heavy corpora over two- and three-letter
    alphabets, where the (left id, right id) tie-break decides most rounds."""
    pytest.importorskip("regex")
    import numpy as np
    from pins import naive_train
    corpora = [workloads.tiny_corpus()[:24_000]]
    rng = np.random.default_rng(31)
    for alphabet in (b"ab", b"abc", b"ab1 "):
        words = [bytes(rng.choice(list(alphabet), size=int(rng.integers(1, 9))).astype(np.uint8))
                 for _ in range(600)]
        corpora.append(b" ".join(words))
    for corpus in corpora:
        got = oracle.train(corpus, 120)
        exp = naive_train(corpus, 120)
        assert got == exp, (corpus[:40], next((i, g, e) for i, (g, e) in enumerate(zip(got, exp)) if g != e)
                            if got[:len(exp)] != exp[:len(got)] else (len(got), len(exp)))
