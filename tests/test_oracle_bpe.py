"""Pins for the oracle's BPE (E): the pages' worked non-concatenation example,
agreement of three independent loops, the fixpoint invariant, degenerate
vocabularies and hand-worked tie-breaks."""
import random

from oracle.bpe import bpe_heap, bpe_rounds, bpe_textbook
from oracle.encode import decode, encode
from oracle.pretokenize import PATTERN_CL100K, PATTERN_GPT2
from oracle.vocab import Vocab


def _vocab_from_strings(merge_strings):
    """Byte tokens 0..255 and merges given as (left bytes, right bytes)."""
    toks = [bytes([b]) for b in range(256)]
    idx = {t: i for i, t in enumerate(toks)}
    merges = []
    for a, b in merge_strings:
        a, b = a.encode(), b.encode()
        if a + b not in idx:
            idx[a + b] = len(toks)
            toks.append(a + b)
        merges.append((idx[a], idx[b]))
    return Vocab(toks, merges), idx


def test_pipe_line_pipeline_example():
    # TokTier, Sections 1.2 and 3.2: "pipe" alone is one token; appending
    # "line" yields the single token "pipeline", so tok(pipe) + tok(line) is
    # not tok(pipeline).
    v, idx = _vocab_from_strings([("p", "i"), ("p", "e"), ("pi", "pe"), ("l", "i"), ("n", "e"),
                                  ("li", "ne"), ("pipe", "line")])
    for pat in (PATTERN_GPT2, PATTERN_CL100K):
        assert encode(b"pipe", v, pat) == [idx[b"pipe"]]
        assert encode(b"line", v, pat) == [idx[b"line"]]
        assert encode(b"pipeline", v, pat) == [idx[b"pipeline"]]
        assert encode(b"pipe", v, pat) + encode(b"line", v, pat) != encode(b"pipeline", v, pat)
        assert encode(b"pipe line", v, pat) == [idx[b"pipe"], 32, idx[b"line"]]


def test_zero_merges_is_bytes():
    v = Vocab.from_merges([])
    data = "héllo 世界 1234\n".encode()
    assert encode(data, v, PATTERN_GPT2) == list(data)
    assert encode(data, v, PATTERN_CL100K) == list(data)


def test_leftmost_tie_break_and_rank_order():
    v, idx = _vocab_from_strings([("a", "a")])
    mm = v.merge_map
    aa = idx[b"aa"]
    for f in (bpe_textbook, bpe_rounds, bpe_heap):
        assert f([97, 97, 97], mm) == [aa, 97]
        assert f([97, 97, 97, 97], mm) == [aa, aa]
        assert f([98, 97, 97, 97, 98], mm) == [98, aa, 97, 98]
    # lower rank wins wherever it is: (b,c) rank 0 beats (a,b) rank 1
    v2, i2 = _vocab_from_strings([("b", "c"), ("a", "b")])
    for f in (bpe_textbook, bpe_rounds, bpe_heap):
        assert f([97, 98, 99], v2.merge_map) == [97, i2[b"bc"]]


def test_local_minima_are_not_enough():
    # ranks AB=3, BC=5, CD=1 plus BX=2 where X=CD: merging both local minima
    # (AB and CD) at once gives (AB)(CD); the rule gives A(B(CD)).
    v, idx = _vocab_from_strings([("x", "y"), ("c", "d"), ("b", "cd"), ("a", "b"), ("q", "r"), ("b", "c")])
    mm = v.merge_map
    want = [97, idx[b"bcd"]]
    for f in (bpe_textbook, bpe_rounds, bpe_heap):
        assert f([97, 98, 99, 100], mm) == want


def _random_vocab(rnd, alphabet, n_merges):
    toks = [bytes([b]) for b in range(256)]
    idx = {t: i for i, t in enumerate(toks)}
    live = [ord(c) for c in alphabet]
    merges = []
    seen = set()
    tries = 0
    while len(merges) < n_merges and tries < 10 * n_merges:
        tries += 1
        a, b = rnd.choice(live), rnd.choice(live)
        if (a, b) in seen or len(toks[a]) + len(toks[b]) > 6:
            continue
        seen.add((a, b))
        t = toks[a] + toks[b]
        if t not in idx:
            idx[t] = len(toks)
            toks.append(t)
            live.append(idx[t])
        merges.append((a, b))
    return Vocab(toks, merges)


def test_three_loops_agree_on_random_vocabs():
    rnd = random.Random(3)
    n_mono = 0
    for trial in range(300):
        v = _random_vocab(rnd, "abc", rnd.randint(1, 25))
        mono = v.monotone()
        n_mono += mono
        for _ in range(20):
            w = [rnd.choice(b"abc") for _ in range(rnd.randint(0, 24))]
            t = bpe_textbook(w, v.merge_map)
            assert bpe_heap(w, v.merge_map) == t
            if mono:
                assert bpe_rounds(w, v.merge_map) == t
            # fixpoint: no adjacent output pair is a merge
            assert all((x, y) not in v.merge_map for x, y in zip(t, t[1:]))
            assert b"".join(v.token_bytes[i] for i in t) == bytes(w)
    assert n_mono > 50


def test_heap_matches_textbook_on_long_words():
    rnd = random.Random(9)
    v = _random_vocab(rnd, "ab ", 60)
    for n in (200, 1000):
        w = [rnd.choice(b"ab ") for _ in range(n)]
        assert bpe_heap(w, v.merge_map) == bpe_textbook(w, v.merge_map)


def test_decode_roundtrip_and_vocab_checks():
    v, _ = _vocab_from_strings([("h", "e"), ("l", "l"), ("he", "ll"), (" ", "w")])
    data = "hello world héllo\r\n".encode()
    assert decode(encode(data, v, PATTERN_GPT2), v) == data
    import pytest
    from oracle.vocab import VocabError
    with pytest.raises(VocabError):
        Vocab([bytes([b]) for b in range(255)], [])
    with pytest.raises(VocabError):
        Vocab([bytes([b]) for b in range(256)], [(97, 97), (97, 97)])
    with pytest.raises(VocabError):
        Vocab([bytes([b]) for b in range(256)], [(97, 98)])  # result bytes missing


def _pair_barriers(word_bytes, vocab):
    """Positions i (0 < i < len) such that no merge result's bytes contain the
    byte pair (word[i-1], word[i])."""
    held = set()
    for _, res in vocab.merge_map.values():
        t = vocab.token_bytes[res]
        held.update(zip(t, t[1:]))
    return [i for i in range(1, len(word_bytes)) if (word_bytes[i - 1], word_bytes[i]) not in held]


def test_words_split_exactly_where_no_merge_result_holds_the_byte_pair():
    # A merge that joins symbols across the boundary between bytes i-1 and i
    # makes a token whose bytes contain that pair; where no merge result
    # contains it, no merge ever crosses i, the two sides evolve apart, and
    # BPE of the word is the concatenation of BPE of its pieces (any vocabulary,
    # monotone or not).  The library splits long fragments there.
    rnd = random.Random(21)
    n_split = 0
    for trial in range(300):
        v = _random_vocab(rnd, "abcd", rnd.randint(1, 30))
        for _ in range(20):
            w = bytes(rnd.choice(b"abcd") for _ in range(rnd.randint(0, 30)))
            cuts = [0] + _pair_barriers(w, v) + [len(w)]
            n_split += len(cuts) > 2
            whole = bpe_textbook([v.byte_id[x] for x in w], v.merge_map)
            parts = []
            for a, b in zip(cuts, cuts[1:]):
                parts += bpe_textbook([v.byte_id[x] for x in w[a:b]], v.merge_map)
            assert parts == whole, (w, cuts)
    assert n_split > 1000
    # a cut where the pair does occur in a merge result is not safe: pipe|line
    v, idx = _vocab_from_strings([("p", "i"), ("p", "e"), ("pi", "pe"), ("l", "i"), ("n", "e"), ("li", "ne"),
                                  ("pipe", "line")])
    w = b"pipeline"
    assert 4 not in _pair_barriers(w, v)
    assert bpe_textbook(list(w), v.merge_map) == [idx[b"pipeline"]]


def test_pair_barriers_on_a_trained_vocabulary_and_a_long_letter_run():
    import os
    import textgen
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    v = Vocab.load_merges(os.path.join(root, "data", "vocabs", "cl100k_session_100k.merges"))
    run = [p for p in textgen.adversarial_pieces(1005, scale=0.004) if p.isalpha() or p[:-1].isalpha()]
    w = max(run, key=len).strip().encode()
    cuts = [0] + _pair_barriers(w, v) + [len(w)]
    assert len(cuts) > 20
    parts = []
    for a, b in zip(cuts, cuts[1:]):
        parts += bpe_heap([v.byte_id[x] for x in w[a:b]], v.merge_map)
    assert parts == bpe_heap([v.byte_id[x] for x in w], v.merge_map)


def test_ignore_merges_takes_whole_tokens_only_for_whole_fragments():
    # "abc" is a token made by (a, bc), but (a, b) ranks first, so BPE of the
    # bytes gives [ab, c]; with ignore_merges the fragment "abc" is the token
    # "abc" itself (Section 4.2's whole-word lookup), while a fragment that is
    # not a token ("abcc") still goes through BPE
    v, idx = _vocab_from_strings([("a", "b"), ("b", "c"), ("a", "bc")])
    mm = v.merge_map
    assert bpe_textbook(list(b"abc"), mm) == [idx[b"ab"], 99]
    assert encode(b"abc", v, PATTERN_GPT2) == [idx[b"ab"], 99]
    assert encode(b"abc", v, PATTERN_GPT2, ignore_merges=True) == [idx[b"abc"]]
    assert encode(b"abcc abc", v, PATTERN_GPT2, ignore_merges=True) == (
        bpe_textbook(list(b"abcc"), mm) + encode(b" abc", v, PATTERN_GPT2))
    # the pages' pipe / line example: with every piece a token, both readings agree
    v2, idx2 = _vocab_from_strings([("p", "i"), ("p", "e"), ("pi", "pe"), ("l", "i"), ("n", "e"), ("li", "ne"),
                                    ("pipe", "line")])
    for w in (b"pipe", b"line", b"pipeline"):
        assert encode(w, v2, PATTERN_GPT2, ignore_merges=True) == encode(w, v2, PATTERN_GPT2) == [idx2[w]]
    # a fragment with no whole token is unchanged by the flag
    rnd = random.Random(31)
    for _ in range(200):
        vr = _random_vocab(rnd, "abc", rnd.randint(1, 20))
        w = bytes(rnd.choice(b"abc") for _ in range(rnd.randint(1, 12)))
        want = [vr.index[w]] if w in vr.index else bpe_heap(list(w), vr.merge_map)
        assert encode(w, vr, PATTERN_GPT2, ignore_merges=True) == want
