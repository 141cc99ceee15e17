"""Pins for the oracle's pre-tokenizer (G), all four patterns: the committed
split examples, the third-party `regex` module on every short string over an
adversarial alphabet and on generated text, and the partition invariant."""
import itertools
import json
import os
import random

import pytest

import textgen
from oracle.pretokenize import PATTERN_CL100K, PATTERN_DEEPSEEK, PATTERN_GPT2, PATTERN_O200K, pretokenize
from oracle.utf8 import decode_utf8

HERE = os.path.dirname(os.path.abspath(__file__))

GPT2_RE = r"""'s|'t|'re|'ve|'m|'ll|'d| ?\p{L}+| ?\p{N}+| ?[^\s\p{L}\p{N}]+|\s+(?!\S)|\s+"""
CL100K_RE = (r"""(?i:'s|'t|'re|'ve|'m|'ll|'d)|[^\r\n\p{L}\p{N}]?\p{L}+|\p{N}{1,3}"""
             r"""| ?[^\s\p{L}\p{N}]+[\r\n]*|\s*[\r\n]+|\s+(?!\S)|\s+""")

# the o200k-style pattern as include/tok.h states it (this project's own
# definition)
O200K_RE = (r"""[^\r\n\p{L}\p{N}]?[\p{Lu}\p{Lt}]*[\p{Ll}\p{Lm}\p{Lo}]+(?:(?i:'s|'t|'re|'ve|'m|'ll|'d))*"""
            r"""|[^\r\n\p{L}\p{N}]?[\p{Lu}\p{Lt}]+(?:(?i:'s|'t|'re|'ve|'m|'ll|'d))*"""
            r"""|\p{N}{1,3}| ?[^\s\p{L}\p{N}]+[\r\n/]*|\s*[\r\n]+|\s+(?!\S)|\s+""")

# the DeepSeek-style pattern as include/tok.h states it (this project's own
# definition): C = letters of script extensions Han, Hiragana, Katakana, Hangul
CJK_RE = r"[\p{scx=Han}\p{scx=Hiragana}\p{scx=Katakana}\p{scx=Hangul}]"
DEEPSEEK_RE = (r"(?i:'s|'t|'re|'ve|'m|'ll|'d)|[^\r\n\p{L}\p{N}]?(?:(?!" + CJK_RE + r")\p{L})+|(?:(?=" + CJK_RE
               + r")\p{L})+|\p{N}{1,3}| ?[^\s\p{L}\p{N}]+[\r\n]*|\s*[\r\n]+|\s+(?!\S)|\s+")

ALPHABET = "asStlLe1² \t\n\r'.éx́中 ſ/カー한"


def split(s, pat):
    cps, _ = decode_utf8(s.encode())
    return [s[a:b] for a, b in pretokenize(cps, pat)]


def test_pinned_examples():
    n = 0
    with open(os.path.join(HERE, "golden", "pretoken_pins.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            s, g, c = json.loads(line)
            assert split(s, PATTERN_GPT2) == g, s
            assert split(s, PATTERN_CL100K) == c, s
            n += 1
    assert n >= 20


def test_pinned_examples_o200k_style():
    # splits the regex module gave for the o200k-style pattern
    # (tests/golden/make_o200k_pins.py): camelCase splits, contractions as
    # suffixes, caseless letters, the [\r\n/]* tail
    n = 0
    with open(os.path.join(HERE, "golden", "pretoken_pins_o200k.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            s, want = json.loads(line)
            assert split(s, PATTERN_O200K) == want, s
            n += 1
    assert n >= 40


def test_pinned_examples_deepseek_style():
    # splits the regex module gave for the DeepSeek-style pattern
    # (tests/golden/make_deepseek_pins.py): CJK runs apart from other letters
    # and without a prefix, kana with the prolonged sound mark, Hangul
    n = 0
    with open(os.path.join(HERE, "golden", "pretoken_pins_deepseek.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            s, want = json.loads(line)
            assert split(s, PATTERN_DEEPSEEK) == want, s
            n += 1
    assert n >= 40


def test_partition_and_empty():
    assert pretokenize([], PATTERN_GPT2) == []
    s = textgen.mixed_c2(4000, 3)
    for pat in (PATTERN_GPT2, PATTERN_CL100K, PATTERN_O200K, PATTERN_DEEPSEEK):
        parts = split(s, pat)
        assert "".join(parts) == s and all(parts)


def _regex_split(rx, s):
    return rx.findall(s)


def test_brute_force_against_regex_module():
    regex = pytest.importorskip("regex")
    rg, rc, ro = regex.compile(GPT2_RE), regex.compile(CL100K_RE), regex.compile(O200K_RE)
    rd = regex.compile(DEEPSEEK_RE)
    for n in range(1, 4):
        for t in itertools.product(ALPHABET, repeat=n):
            s = "".join(t)
            assert split(s, PATTERN_GPT2) == rg.findall(s), repr(s)
            assert split(s, PATTERN_CL100K) == rc.findall(s), repr(s)
            assert split(s, PATTERN_O200K) == ro.findall(s), repr(s)
            assert split(s, PATTERN_DEEPSEEK) == rd.findall(s), repr(s)
    rnd = random.Random(11)
    for _ in range(5000):
        s = "".join(rnd.choice(ALPHABET) for _ in range(rnd.randint(4, 16)))
        assert split(s, PATTERN_GPT2) == rg.findall(s), repr(s)
        assert split(s, PATTERN_CL100K) == rc.findall(s), repr(s)
        assert split(s, PATTERN_O200K) == ro.findall(s), repr(s)
        assert split(s, PATTERN_DEEPSEEK) == rd.findall(s), repr(s)


def test_brute_force_five_code_points_against_regex_module(oracle_pool):
    # every string of 1..5 code points over the adversarial alphabet (about
    # 580,000 strings), the oracle on all host cores
    regex = pytest.importorskip("regex")
    from conftest import BRUTE_ALPHABET
    strs = ["".join(t) for n in range(1, 6) for t in itertools.product(BRUTE_ALPHABET, repeat=n)]
    enc = [s.encode() for s in strs]
    for pat, rx in ((PATTERN_GPT2, regex.compile(GPT2_RE)), (PATTERN_CL100K, regex.compile(CL100K_RE)),
                    (PATTERN_O200K, regex.compile(O200K_RE)), (PATTERN_DEEPSEEK, regex.compile(DEEPSEEK_RE))):
        got = oracle_pool.starts_many(enc, pat)
        for s, g in zip(strs, got):
            want, pos = [], 0
            for m in rx.findall(s):
                want.append(pos)
                pos += len(m.encode())
            assert g == want, repr(s)


def test_generated_text_against_regex_module():
    regex = pytest.importorskip("regex")
    rg, rc, ro = regex.compile(GPT2_RE), regex.compile(CL100K_RE), regex.compile(O200K_RE)
    rd = regex.compile(DEEPSEEK_RE)
    texts = [textgen.code_ascii(8000, 1), textgen.mixed_c2(20000, 2), textgen.agentic_session(20000, 3)]
    texts += textgen.adversarial_pieces(5, scale=0.002)
    for s in texts:
        assert split(s, PATTERN_GPT2) == rg.findall(s)
        assert split(s, PATTERN_CL100K) == rc.findall(s)
        assert split(s, PATTERN_O200K) == ro.findall(s)
        assert split(s, PATTERN_DEEPSEEK) == rd.findall(s)
