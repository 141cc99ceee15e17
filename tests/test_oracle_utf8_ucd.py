"""Pins for the oracle's UTF-8 decoder and class table.

UTF-8: against CPython's strict codec (an independent implementation of RFC
3629) on every 1- and 2-byte sequence, on every lead byte combined with the
boundary values of each continuation position, and on random sequences.
Classes: against the third-party `regex` module for every code point (where
it is installed), and against fixed values from the Unicode standard."""
import itertools
import random

import pytest

from oracle.ucd import classify
from oracle.utf8 import Utf8Error, decode_utf8


def _py(data):
    try:
        return ("ok", [ord(c) for c in data.decode("utf-8")])
    except UnicodeDecodeError as e:
        return ("err", e.start)


def _ours(data):
    try:
        cps, offs = decode_utf8(data)
        assert len(offs) == len(cps) + 1 and offs[-1] == len(data)
        return ("ok", cps)
    except Utf8Error as e:
        return ("err", e.offset)


def test_utf8_all_short_sequences():
    for n in (1, 2):
        for t in itertools.product(range(256), repeat=n):
            d = bytes(t)
            assert _ours(d) == _py(d), d


def test_utf8_boundary_values():
    edges = [0x00, 0x41, 0x7F, 0x80, 0x8F, 0x90, 0x9F, 0xA0, 0xBF, 0xC0, 0xC2, 0xE0, 0xED, 0xF0, 0xF4, 0xFF]
    for lead in range(0x80, 0x100):
        for rest in itertools.product(edges, repeat=3):
            for k in (1, 2, 3, 4):
                d = bytes([lead]) + bytes(rest[:k - 1]) + b"a"
                assert _ours(d) == _py(d), d
                d2 = b"xy" + d
                assert _ours(d2) == _py(d2), d2


def test_utf8_random_and_offsets():
    rnd = random.Random(7)
    for _ in range(20000):
        d = bytes(rnd.choice([rnd.randrange(256), rnd.randrange(0x80, 0xC0), 0xE4, 0xF0, 0x61])
                  for _ in range(rnd.randint(0, 12)))
        assert _ours(d) == _py(d), d
    s = "aé中\U0001F600z"
    cps, offs = decode_utf8(s.encode())
    assert cps == [ord(c) for c in s]
    assert offs == [0, 1, 3, 6, 10, 11]


def test_classes_fixed_values():
    assert classify(0x20) == "W" and classify(0x0A) == "W" and classify(0xA0) == "W"
    assert classify(0x3000) == "W" and classify(0x85) == "W" and classify(0x2028) == "W"
    for cp in (0x1C, 0x1D, 0x1E, 0x1F, 0x200B, 0x180E):  # not White_Space
        assert classify(cp) == "O"
    assert classify(ord("A")) == "L" and classify(0x4E00) == "L" and classify(0x17F) == "L"
    assert classify(0x1C89) == "L"  # added in Unicode 16.0
    assert classify(ord("7")) == "N" and classify(0xB2) == "N" and classify(0xBD) == "N"
    assert classify(0x2167) == "N" and classify(0x1D7D8) == "N"
    assert classify(0x301) == "O" and classify(0x27) == "O" and classify(0x1F600) == "O"
    assert classify(0x10FFFF) == "O" and classify(0xE000) == "O"
    ws = [cp for cp in range(0x3001) if classify(cp) == "W"]
    assert len(ws) == 25


def test_classes_match_regex_module_everywhere():
    regex = pytest.importorskip("regex")
    pl, pn, ps = regex.compile(r"\p{L}"), regex.compile(r"\p{N}"), regex.compile(r"\s")
    for cp in range(0x110000):
        if 0xD800 <= cp <= 0xDFFF:
            continue
        ch = chr(cp)
        want = "L" if pl.match(ch) else "N" if pn.match(ch) else "W" if ps.match(ch) else "O"
        assert classify(cp) == want, hex(cp)


def test_cjk_letters_match_regex_module_everywhere():
    # the DeepSeek-style pattern's CJK letters: letters whose script
    # extensions include Han, Hiragana, Katakana or Hangul
    regex = pytest.importorskip("regex")
    from oracle.ucd import is_cjk
    pc = regex.compile(r"(?=[\p{scx=Han}\p{scx=Hiragana}\p{scx=Katakana}\p{scx=Hangul}])\p{L}")
    for cp in range(0x110000):
        if 0xD800 <= cp <= 0xDFFF:
            continue
        assert is_cjk(cp) == bool(pc.match(chr(cp))), hex(cp)
    # fixed values: Han, kana with the prolonged sound mark, Hangul; not
    # Bopomofo, Latin, digits or CJK punctuation
    for cp in (0x4E2D, 0x3005, 0x30AB, 0x30FC, 0x3072, 0xD55C, 0xFF71, 0x20000, 0x3400):
        assert is_cjk(cp), hex(cp)
    for cp in (0x3105, ord("a"), 0xE9, ord("1"), 0x3002, 0x3001, 0x4E00 - 1):
        assert not is_cjk(cp), hex(cp)

