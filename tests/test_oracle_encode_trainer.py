"""Pins for the whole oracle pipeline and its trainer: round trip, the
fragment-independence definition of F = E* . G (TokTier, Appendix A.1), the
splice theorem (Appendix A.2), trainer determinism and a hand-worked
training run."""
import os
import random

import pytest

import textgen
from oracle.bpe import bpe_heap, bpe_textbook
from oracle.encode import decode, encode, encode_with_offsets, pretoken_byte_spans
from oracle.pretokenize import PATTERN_CL100K, PATTERN_GPT2
from oracle.trainer import TrainError, fragment_counts, train, train_from_counts, train_naive
from oracle.utf8 import Utf8Error
from oracle.vocab import Vocab, read_merges

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def small_vocab():
    corpus = textgen.mixed_c2(200_000, 77).encode()
    return Vocab.from_merges(train(corpus, PATTERN_GPT2, 600))


def test_roundtrip_and_fragment_independence(small_vocab):
    v = small_vocab
    for pat in (PATTERN_GPT2, PATTERN_CL100K):
        for s in (textgen.mixed_c2(30000, 5), textgen.agentic_session(20000, 6)):
            data = s.encode()
            ids = encode(data, v, pat)
            assert decode(ids, v) == data
            # F = E* . G: the encoding is the concatenation of per-fragment encodings
            per = []
            for a, b in pretoken_byte_spans(data, pat):
                per.extend(encode(data[a:b], v, pat))
            assert per == ids
            # the textbook loop gives the same ids
            assert encode(data, v, pat, bpe=bpe_textbook) == ids


def test_splice_theorem(small_vocab):
    # Appendix A.2: if no fragment crosses the cut and both sides' fragments
    # equal the whole text's, the two encodings concatenate to the whole one.
    v = small_vocab
    rnd = random.Random(1)
    s = textgen.agentic_session(6000, 8)
    data = s.encode()
    for pat in (PATTERN_GPT2, PATTERN_CL100K):
        whole = encode(data, v, pat)
        spans = pretoken_byte_spans(data, pat)
        cuts = [a for a, _ in spans[1:]]
        certified = 0
        for c in rnd.sample(cuts, 60):
            left = pretoken_byte_spans(data[:c], pat)
            right = [(a + c, b + c) for a, b in pretoken_byte_spans(data[c:], pat)]
            if left + right == spans:
                certified += 1
                assert encode(data[:c], v, pat) + encode(data[c:], v, pat) == whole
        assert certified > 20


def test_token_offsets(small_vocab):
    # each token's bytes sit at its offset; every fragment start is a token
    # start (fragments are encoded independently, Appendix A.1)
    v = small_vocab
    for pat in (PATTERN_GPT2, PATTERN_CL100K):
        data = textgen.agentic_session(8000, 9).encode()
        ids, offs = encode_with_offsets(data, v, pat)
        assert len(offs) == len(ids) and (not offs or offs[0] == 0)
        ends = offs[1:] + [len(data)]
        for i, a, b in zip(ids, offs, ends):
            assert data[a:b] == v.token_bytes[i]
        assert {a for a, _ in pretoken_byte_spans(data, pat)} <= set(offs)
    assert encode_with_offsets(b"", v, PATTERN_GPT2) == ([], [])


def test_utf8_error_offset():
    v = Vocab.from_merges([])
    with pytest.raises(Utf8Error) as e:
        encode(b"abc\xe4\xb8", v, PATTERN_GPT2)
    assert e.value.offset == 3


def test_trainer_hand_example():
    # one fragment "aaabdaaabac": (a,a) occurs 4 times -> merge 0; then
    # (a,b) and (aa,a) both occur twice and the smaller pair (97,98) wins;
    # then (aa,ab) occurs twice.
    counts = fragment_counts(b"aaabdaaabac", PATTERN_GPT2)
    assert dict(counts) == {b"aaabdaaabac": 1}
    m = train_from_counts(counts, 3, min_count=2)
    assert m == [(97, 97), (97, 98), (256, 257)]
    v = Vocab.from_merges(m)
    assert v.token_bytes[258] == b"aaab"
    with pytest.raises(TrainError):
        train_from_counts(counts, 4, min_count=2)


def test_trainer_incremental_equals_naive_and_deterministic():
    corpus = textgen.code_ascii(30000, 4).encode()
    counts = fragment_counts(corpus, PATTERN_GPT2)
    a = train_from_counts(counts, 150, min_count=1)
    assert a == train_naive(counts, 150, min_count=1)
    assert a == train_from_counts(fragment_counts(corpus, PATTERN_GPT2), 150, min_count=1)


def test_committed_small_vocab_reproduces():
    # the committed 1k vocabulary is exactly what the trainer produces
    import sys
    sys.path.insert(0, os.path.join(ROOT, "data"))
    import make_vocabs
    pattern, kind, mib, seed, n = make_vocabs.VOCABS["gpt2_code_1k"]
    total = {}
    for d in range(mib):
        c = make_vocabs._doc_counts((kind, seed * 1000 + d, pattern))
        for k, val in c.items():
            total[k] = total.get(k, 0) + val
    merges = train_from_counts(total, n, min_count=2)
    assert merges == read_merges(os.path.join(ROOT, "data", "vocabs", "gpt2_code_1k.merges"))
    v = Vocab.from_merges(merges)
    assert v.monotone()
    data = textgen.code_ascii(16384, 1001).encode()
    ids = encode(data, v, PATTERN_GPT2)
    assert decode(ids, v) == data and len(ids) < len(data) // 2
    assert ids == encode(data, v, PATTERN_GPT2, bpe=bpe_heap)


def test_windowed_oracle_equals_whole_text(small_vocab):
    # the full-size parity tests run the oracle window by window, cut at
    # certified cuts (tests/oracle_par.py); on texts the oracle finishes in
    # seconds the windows' ids and shifted fragment starts equal the whole
    # text's, for both patterns, including a window that is one long run
    from oracle.encode import encode_with_spans
    from oracle_par import is_cut, windows
    v = small_vocab
    texts = [textgen.adversarial(300_000, 1005, scale=0.02).encode(), textgen.agentic_session(60_000, 8).encode(),
             b"abc" * 5000 + b".x" + b"9" * 7000 + b"-" + "é".encode() * 900 + b"a's'" + b"q" * 3000]
    for data in texts:
        cuts = windows(data, 4096)
        assert len(cuts) > 3 and cuts[0] == 0 and cuts[-1] == len(data)
        assert all(is_cut(data, c) for c in cuts[1:-1])
        for pat in (PATTERN_GPT2, PATTERN_CL100K):
            ids, spans = encode_with_spans(data, v, pat)
            got_ids, got_starts = [], []
            for a, b in zip(cuts, cuts[1:]):
                i, s = encode_with_spans(data[a:b], v, pat)
                got_ids += i
                got_starts += [a + x for x, _ in s]
            assert got_ids == ids
            assert got_starts == [x for x, _ in spans]
