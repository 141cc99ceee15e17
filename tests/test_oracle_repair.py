"""Pins for the session-repair oracle (TokTier, Section 3.3; the splice
theorem, Appendix A.2): repairing an append must give exactly the encoding of
the whole text, on random short strings over an alphabet that exercises every
boundary rule of both patterns, on the pages' pipe/line example, and on
agent sessions cut at random places."""
import random

import pytest

import textgen
from oracle.encode import encode_with_offsets
from oracle.pretokenize import PATTERN_CL100K, PATTERN_GPT2
from oracle.repair import last_cut, repair_append
from oracle.trainer import train
from oracle.vocab import Vocab

ALPHABET = ["a", "b", "Z", "é", "中", "1", "2", "٣", " ", "  ", "\n", "\r\n", "\t", "'", "'s", "'LL", ".", "!", " ",
            "́", "x1", "ſ"]


@pytest.fixture(scope="module")
def vocab():
    corpus = (textgen.mixed_c2(120_000, 31) + textgen.agentic_session(60_000, 32)).encode()
    return Vocab.from_merges(train(corpus, PATTERN_CL100K, 500))


def _check(v, pat, old, delta):
    old_ids, old_offs = encode_with_offsets(old, v, pat)
    ids, offs, n = repair_append(old, old_ids, old_offs, delta, v, pat)
    want_ids, want_offs = encode_with_offsets(old + delta, v, pat)
    assert (ids, offs) == (want_ids, want_offs), (old, delta)
    assert 0 <= n <= len(old) + len(delta)
    return n


def test_random_short_appends(vocab):
    rng = random.Random(5)
    for pat in (PATTERN_GPT2, PATTERN_CL100K):
        for _ in range(4000):
            old = "".join(rng.choice(ALPHABET) for _ in range(rng.randrange(0, 9))).encode()
            delta = "".join(rng.choice(ALPHABET) for _ in range(rng.randrange(0, 5))).encode()
            _check(vocab, pat, old, delta)


def test_pipe_line_example():
    # the pages' example (Section 3.2): "pipe" + "line" must not stay two tokens
    toks = [bytes([b]) for b in range(256)]
    merges = []

    def add(a, b):
        ia, ib = toks.index(a), toks.index(b)
        if a + b not in toks:
            toks.append(a + b)
        merges.append((ia, ib))
    for a, b in ((b"p", b"i"), (b"p", b"e"), (b"pi", b"pe"), (b"l", b"i"), (b"n", b"e"), (b"li", b"ne"),
                 (b"pipe", b"line")):
        add(a, b)
    v = Vocab.from_merges(merges)
    for pat in (PATTERN_GPT2, PATTERN_CL100K):
        old, delta = b"the pipe", b"line"
        n = _check(v, pat, old, delta)
        assert n == len(b" pipeline")  # re-encoded from the space before "pipe"
        ids, _ = encode_with_offsets(old + delta, v, pat)
        assert v.token_bytes[ids[-1]] == b"pipeline"


def test_cut_position_rule():
    assert last_cut(b"") == 0 and last_cut(b"abc") == 0
    assert last_cut(b"ab cd") == 2          # letter, then space
    assert last_cut(b"x123") == 1           # letter, then number
    assert last_cut(b"x123.") == 4          # number, then '.'
    assert last_cut("é中1".encode()) == 5    # L L N: the cut is at the number (byte 5)
    assert last_cut(b"a  \n") == 1


def test_sessions_cut_anywhere(vocab):
    rng = random.Random(9)
    s = textgen.agentic_session(30_000, 77).encode()
    for pat in (PATTERN_GPT2, PATTERN_CL100K):
        for _ in range(12):
            a = rng.randrange(0, len(s) - 2000)
            b = a + rng.randrange(1, 1500)
            old, delta = s[:a], s[a:b]
            # cut only at code point boundaries (the text is valid UTF-8 on both sides)
            try:
                old.decode("utf-8")
                delta.decode("utf-8")
            except UnicodeDecodeError:
                continue
            n = _check(vocab, pat, old, delta)
            assert n <= len(delta) + 4096  # the cut sits near the end of old
