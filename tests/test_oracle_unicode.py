"""Pins of the oracle's Unicode classes against the regex library and the
Unicode database shipped with Python."""
import os
import unicodedata

import pytest

import oracle


def test_classes_match_regex_library():
    regex = pytest.importorskip("regex")
    pl, pn, ps = regex.compile(r"\p{L}"), regex.compile(r"\p{N}"), regex.compile(r"\s")
    for c in range(0x110000):
        ch = chr(c)
        exp = 1 if pl.match(ch) else 2 if pn.match(ch) else 3 if ps.match(ch) else 0
        assert oracle.cp_class(c) == exp, hex(c)


def test_classes_agree_with_unicodedata_where_assigned_in_both():
    # Python's unicodedata may lag the regex module's Unicode version; compare
    # only code points assigned in Python's database.
    for c in range(0x110000):
        cat = unicodedata.category(chr(c))
        if cat == "Cn":
            continue
        k = oracle.cp_class(c)
        if cat[0] == "L":
            assert k == 1, hex(c)
        elif cat[0] == "N":
            assert k == 2, hex(c)


def test_white_space_is_exactly_25_code_points():
    ws = [c for c in range(0x110000) if oracle.cp_class(c) == 3]
    assert ws == [0x9, 0xA, 0xB, 0xC, 0xD, 0x20, 0x85, 0xA0, 0x1680] + list(range(0x2000, 0x200B)) + \
        [0x2028, 0x2029, 0x202F, 0x205F, 0x3000]


def test_header_is_current():
    """The committed range table matches what the generator would write now."""
    pytest.importorskip("regex")
    import hashlib
    import importlib.util
    here = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle")
    spec = importlib.util.spec_from_file_location("gen", os.path.join(here, "gen_unicode_ranges.py"))
    gen = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(gen)
    digest = hashlib.sha256(bytes(gen.class_of_all())).hexdigest()
    with open(os.path.join(here, "unicode_ranges.h")) as f:
        assert digest in f.read()
