"""The BPE kernel's grid engine: when the fragments longer than 256 bytes
hold at least 32 KiB, a group of the kernel's CTAs encodes all of them at
once, meeting at grid barriers between the steps of each sweep; with fewer
bytes, the same CTAs encode one fragment each.

Parity: ids against the oracle, id for id, on texts made of such fragments
(whitespace, newline, digit and letter runs of 200 bytes to 100 KB, repeated
symbols whose merges pair up from the left end of the run, 2-byte letters)
under both patterns, as one text and as batch items; the same texts with the
vocabulary's merges ignored; under the o200k-style pattern, with token
offsets; long-fragment bytes on both sides of the 32 KiB switch; about 4,000
long fragments at once; long fragments of fewer bytes in all; and a
non-monotone vocabulary, which keeps the one-CTA engine.  The wait limit: a
barrier that never completes (made on the host with tok_debug_grid_wait) ends
the call with TOK_ETIMEOUT after the limit, and the handle then encodes
normally."""
import os
import random

import pytest

import textgen
from oracle.encode import encode, encode_with_offsets
from oracle.pretokenize import PATTERN_CL100K, PATTERN_GPT2, PATTERN_O200K
from oracle.vocab import Vocab

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
VOC = os.path.join(ROOT, "data", "vocabs")
VOCABS = {PATTERN_GPT2: "gpt2_session_100k", PATTERN_CL100K: "cl100k_session_100k",
          PATTERN_O200K: "cl100k_session_100k"}


@pytest.fixture(scope="module")
def pkg():
    from exact_bpe_tokenization_utf_gb300 import _build
    _build.build()
    import exact_bpe_tokenization_utf_gb300 as p
    return p


_vocabs = {}


def vocab(pattern):
    name = VOCABS[pattern]
    if name not in _vocabs:
        _vocabs[name] = Vocab.load_merges(os.path.join(VOC, name + ".merges"))
    return _vocabs[name]


def tokenizer(pkg, pattern, **kw):
    return pkg.Tokenizer.from_merges_file(os.path.join(VOC, VOCABS[pattern] + ".merges"), pattern, **kw)


def long_text(seed, scale=0.1, n_mid=150):
    """The adversarial components at `scale`, and n_mid runs of 200..5000
    bytes of several kinds between short words, shuffled."""
    r = random.Random(seed)
    kinds = [lambda n: " " * n, lambda n: "\n" * n, lambda n: " \t" * (n // 2),
             lambda n: "".join(r.choice("0123456789") for _ in range(n)), lambda n: "7" * n,
             lambda n: "ab" * (n // 2), lambda n: "é" * (n // 2),
             lambda n: "".join(r.choice("abcdefgh") for _ in range(n)), lambda n: "a" * n]
    parts = textgen.adversarial_pieces(seed, scale)
    for _ in range(n_mid):
        parts.append(r.choice(kinds)(r.randint(200, 5000)) + r.choice(["x", "!", " y", "1", ". "]))
    r.shuffle(parts)
    return "".join(parts).encode()


@pytest.mark.parametrize("pattern", [PATTERN_GPT2, PATTERN_CL100K])
def test_many_long_fragments_match_the_oracle(pkg, pattern):
    v = vocab(pattern)
    assert v.monotone()
    tok = tokenizer(pkg, pattern)
    try:
        for seed in (1, 2):
            data = long_text(seed)
            assert tok.encode(data).tolist() == encode(data, v, pattern), seed
        # one run of each kind alone, just past the size at which the grid
        # engine takes over and well beyond it
        for n in (32 * 1024 + 5, 100_003):
            for s in (" " * n + "x", "\n" * n, "9" * n + " ", "ab" * (n // 2), "é" * (n // 2)):
                data = s.encode()
                assert tok.encode(data).tolist() == encode(data, v, pattern), (n, s[:3])
    finally:
        tok.close()


def test_o200k_style_long_fragments_with_offsets(pkg):
    pattern = PATTERN_O200K
    v = vocab(pattern)
    tok = tokenizer(pkg, pattern)
    try:
        data = long_text(6, n_mid=60)
        ids, offs = tok.encode_with_offsets(data)
        assert (ids.tolist(), offs.tolist()) == encode_with_offsets(data, v, pattern)
    finally:
        tok.close()


@pytest.mark.parametrize("pattern", [PATTERN_GPT2, PATTERN_CL100K])
def test_both_sides_of_the_grid_engine_switch(pkg, pattern):
    # one long space run (a single fragment before "x") of 32 KiB - 1, 32 KiB
    # and 32 KiB + 1 bytes in a text of 40 KB or more; the fragment that ends
    # the run keeps the space before "x", so the run's piece is one byte
    # shorter than the run
    v = vocab(pattern)
    tok = tokenizer(pkg, pattern)
    try:
        filler = textgen.agentic_session(8_000, 77)
        for m in (32 * 1024 - 1, 32 * 1024, 32 * 1024 + 1, 32 * 1024 + 2):
            data = (filler + " " * m + "x" + filler).encode()
            assert tok.encode(data).tolist() == encode(data, v, pattern), m
    finally:
        tok.close()


def test_thousands_of_long_fragments(pkg):
    # about 4,000 fragments of 257..600 bytes (runs of spaces, newlines,
    # digits, letters and dashes, each a single fragment that no byte-pair
    # boundary cuts): every grid-engine CTA scans all their lengths, the
    # coordinates are looked up among thousands of offsets
    pattern = PATTERN_GPT2
    v = vocab(pattern)
    tok = tokenizer(pkg, pattern)
    try:
        r = random.Random(12)
        runs = [" ", "\n", "7", "a", "-"]
        parts = []
        for _ in range(4000):
            ch = r.choice(runs)
            parts.append(ch * r.randint(258, 600) + r.choice(["x", ";", "Q"]))
        data = "".join(parts).encode()
        assert tok.encode(data).tolist() == encode(data, v, pattern)
    finally:
        tok.close()


def test_long_fragments_in_batch_items(pkg):
    pattern = PATTERN_GPT2
    v = vocab(pattern)
    tok = tokenizer(pkg, pattern)
    try:
        data = long_text(3, n_mid=40)
        cuts = sorted(random.Random(3).sample(range(1, len(data)), 7))
        items = [data[a:b] for a, b in zip([0] + cuts, cuts + [len(data)])]
        items.insert(2, b"")
        ids, off = tok.encode_batch(items)
        for j, it in enumerate(items):
            assert ids[off[j]:off[j + 1]].tolist() == encode(it, v, pattern), j
    finally:
        tok.close()


def test_long_fragments_with_merges_ignored(pkg):
    pattern = PATTERN_CL100K
    v = vocab(pattern)
    tok = tokenizer(pkg, pattern, ignore_merges=True)
    try:
        data = long_text(4, n_mid=40)
        assert tok.encode(data).tolist() == encode(data, v, pattern, ignore_merges=True)
    finally:
        tok.close()


@pytest.mark.parametrize("pattern", [PATTERN_GPT2, PATTERN_CL100K])
def test_few_long_fragment_bytes_take_one_cta_each(pkg, pattern):
    # a 200 KB session with eight runs of 300..3000 bytes: below 32 KiB of
    # long fragments, in a text long enough for the grid engine
    v = vocab(pattern)
    tok = tokenizer(pkg, pattern)
    try:
        r = random.Random(5)
        parts = [textgen.agentic_session(25_000, 60 + j) for j in range(8)]
        runs = [" " * 3000, "\n" * 2000, "7" * 1500, "ab" * 400, "é" * 300, "x" * 257, "  " * 1000, "9" * 300]
        data = "".join(p + run + "!" for p, run in zip(parts, runs)).encode()
        assert tok.encode(data).tolist() == encode(data, v, pattern)
    finally:
        tok.close()


def test_non_monotone_vocabulary_keeps_the_cta_engine(pkg):
    # "abc" is made by (ab,c) at rank 1 and again by (a,bc) at rank 4, after
    # (abc,d) used it at rank 2; three 12000-letter words: 36 KB of long fragments
    toks = [bytes([b]) for b in range(256)] + [b"ab", b"abc", b"abcd", b"bc", b"cd", b"dd"]
    ix = {t: i for i, t in enumerate(toks)}
    merges = [(ix[b"a"], ix[b"b"]), (ix[b"ab"], ix[b"c"]), (ix[b"abc"], ix[b"d"]), (ix[b"b"], ix[b"c"]),
              (ix[b"a"], ix[b"bc"]), (ix[b"c"], ix[b"d"]), (ix[b"d"], ix[b"d"])]
    v = Vocab(toks, merges)
    assert not v.monotone()
    tok = pkg.Tokenizer(toks, merges, PATTERN_GPT2)
    try:
        r = random.Random(8)
        data = " ".join("".join(r.choice("abcd") for _ in range(12000)) for _ in range(3)).encode()
        assert tok.encode(data).tolist() == encode(data, v, PATTERN_GPT2)
    finally:
        tok.close()


def test_grid_barrier_wait_limit(pkg):
    import time
    pattern = PATTERN_GPT2
    v = vocab(pattern)
    L = pkg.lib()
    tok = tokenizer(pkg, pattern)
    try:
        data = (" " * 40_000 + "x" + "7" * 30_000).encode()
        want = encode(data, v, pattern)
        assert tok.encode(data).tolist() == want
        # every barrier waits for one CTA more than the grid has: each wait
        # runs out after 50 ms and the call reports it
        assert L.tok_debug_grid_wait(tok._h, 1, 50) == pkg.TOK_OK
        t0 = time.monotonic()
        with pytest.raises(pkg.TokError) as e:
            tok.encode(data)
        assert e.value.code == pkg.TOK_ETIMEOUT
        assert time.monotonic() - t0 < 5.0
        # a text without long fragments has no barrier to wait at
        small = textgen.agentic_session(20_000, 9).encode()
        assert tok.encode(small).tolist() == encode(small, v, pattern)
        # back to normal: the context and the handle are intact
        assert L.tok_debug_grid_wait(tok._h, 0, 0) == pkg.TOK_OK
        assert tok.encode(data).tolist() == want
        assert L.tok_debug_grid_wait(None, 0, 0) == pkg.TOK_EINVAL
    finally:
        tok.close()
