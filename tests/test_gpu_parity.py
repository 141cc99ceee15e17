"""GPU parity: the CUDA library through its C ABI against the oracle.

Integer work, so the bar is bit-exact: every fragment start and every token
id must equal the oracle's, on every workload at its full size (the 16 KiB,
1 MiB and 1M-character texts, all 64 items of the batch, the whole 8 MiB
adversarial text under both patterns).  The large ones run the oracle on all
host cores (tests/oracle_par.py)."""
import itertools
import os
import random

import numpy as np
import pytest

import textgen
from conftest import BRUTE_ALPHABET
from oracle.encode import encode, encode_with_offsets, pretoken_byte_spans
from oracle.repair import repair_append as oracle_repair_append
from oracle.pretokenize import PATTERN_CL100K, PATTERN_DEEPSEEK, PATTERN_GPT2, PATTERN_O200K
from oracle.utf8 import Utf8Error
from oracle.vocab import Vocab

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
VOC = os.path.join(ROOT, "data", "vocabs")

ALPHABET = "asStlLe1² \t\n\r'.éx́中 ſ/カー한"


@pytest.fixture(scope="session")
def pkg():
    from exact_bpe_tokenization_utf_gb300 import _build
    _build.build()
    import exact_bpe_tokenization_utf_gb300 as p
    return p


_cache = {}


def pair(pkg, name, pattern):
    """(oracle vocabulary, GPU tokenizer) for a committed vocabulary."""
    key = (name, pattern)
    if key not in _cache:
        path = os.path.join(VOC, name + ".merges")
        if not os.path.exists(path):
            pytest.skip("vocabulary %s not built" % name)
        _cache[key] = (Vocab.load_merges(path), pkg.Tokenizer.from_merges_file(path, pattern))
    return _cache[key]


def oracle_starts(data, pattern):
    return [a for a, _ in pretoken_byte_spans(data, pattern)]


# --- pre-tokenizer ----------------------------------------------------------

ALL_PATTERNS = [PATTERN_GPT2, PATTERN_CL100K, PATTERN_O200K, PATTERN_DEEPSEEK]


@pytest.mark.parametrize("pattern", ALL_PATTERNS)
def test_pretokenize_brute_force(pkg, pattern):
    tok = pkg.Tokenizer.from_merges([], pattern)
    items = ["".join(t) for n in range(1, 4) for t in itertools.product(ALPHABET, repeat=n)]
    rnd = random.Random(pattern)
    items += ["".join(rnd.choice(ALPHABET) for _ in range(rnd.randint(4, 40))) for _ in range(4000)]
    enc = [s.encode() for s in items]
    got = tok.pretokenize_batch(enc)
    for s, b, g in zip(items, enc, got):
        assert g == oracle_starts(b, pattern), repr(s)


@pytest.mark.parametrize("pattern", ALL_PATTERNS)
def test_pretokenize_brute_force_five_code_points(pkg, oracle_pool, pattern):
    # every string of 1..5 code points over the adversarial alphabet, in one
    # batch call, against the oracle's fragment starts
    tok = pkg.Tokenizer.from_merges([], pattern)
    enc = ["".join(t).encode() for n in range(1, 6) for t in itertools.product(BRUTE_ALPHABET, repeat=n)]
    want = oracle_pool.starts_many(enc, pattern)
    got = tok.pretokenize_batch(enc)
    assert len(got) == len(want)
    bad = [(b, g, w) for b, g, w in zip(enc, got, want) if g != w]
    assert not bad, bad[:5]


@pytest.mark.parametrize("pattern", ALL_PATTERNS)
def test_pretokenize_runs_across_chunks(pkg, pattern):
    # runs far longer than a 1 KiB chunk: whitespace, digits, letters, CR/LF
    tok = pkg.Tokenizer.from_merges([], pattern)
    text = textgen.adversarial(600_000, 1005, scale=0.05).encode()
    assert list(tok.pretokenize(text)) == oracle_starts(text, pattern)
    parts = [b"x;" + b"\n" * 9000 + b" " * 5000 + b"\n" * 3 + b"  y",
             b"a" + b"\r\n" * 5000 + b" " * 3,
             b"1" * 12347 + b"z" + b"2" * 8191,
             b" " * 8192,
             b"'s" * 3000 + b"'" + b" " * 4095 + b"'ll",
             b"x." + b"\n/" * 4000 + b".abc" + b"\r\n" * 700 + b"/" * 900 + b"\n/x",
             b"camelCase" * 500 + b"ABC" * 700 + b"x's" * 400]
    for p in parts:
        assert list(tok.pretokenize(p)) == oracle_starts(p, pattern)
    got = tok.pretokenize_batch(parts)
    for p, g in zip(parts, got):
        assert g == oracle_starts(p, pattern)


def _runs_at_chunk_edges(kinds, lengths, offsets, chunk=1024):
    """One text in which each run (kind * length) is placed so that a chunk
    edge falls at each offset from the run's start (before it, inside it,
    just after it); filler of letters and punctuation between runs."""
    out = bytearray()
    filler = b"ab.c,"
    for kind in kinds:
        for k in lengths:
            run = kind * k
            for d in offsets:
                # pad so that the run starts d bytes before an edge
                target = (-d) % chunk
                pad = (target - len(out)) % chunk
                if pad < 2:
                    pad += chunk
                out += (filler * (pad // len(filler) + 1))[:pad - 1] + b"."
                out += run
    out += b"Z"
    return bytes(out)


@pytest.mark.parametrize("pattern", ALL_PATTERNS)
def test_runs_at_every_offset_of_a_chunk_edge(pkg, pattern):
    # the run states at a chunk's edges come from the window when a run ends
    # within it and from the text beyond it otherwise: runs of CR/LF, digits,
    # spaces, mixed whitespace and apostrophes around the window's reach, and
    # (o200k-style) tails of CR/LF and '/' after a symbol, case changes
    tok = pkg.Tokenizer.from_merges([], pattern)
    kinds = [b"\r\n", b"7", b" ", b"\t\n ", "\u0663".encode(), b"'s", b"\n/", b"aB", b"\n\n /"]
    text = _runs_at_chunk_edges(kinds, [1, 2, 5, 11, 12, 13, 14, 17], range(-3, 20))
    assert list(tok.pretokenize(text)) == oracle_starts(text, pattern)
    name = "gpt2_session_100k" if pattern == PATTERN_GPT2 else "cl100k_session_100k"
    v, tk = pair(pkg, name, pattern)
    small = _runs_at_chunk_edges(kinds, [1, 6, 13, 17], range(-2, 18, 3))
    assert tk.encode(small).tolist() == encode(small, v, pattern)


# --- whole encode at full size -------------------------------------------

def test_encode_code_16k_1k_merges(pkg):
    v, tok = pair(pkg, "gpt2_code_1k", PATTERN_GPT2)
    data = textgen.code_ascii(16384, 1001).encode()
    assert tok.encode(data).tolist() == encode(data, v, PATTERN_GPT2)


def test_encode_mixed_1mib_50k_merges(pkg):
    v, tok = pair(pkg, "gpt2_mixed_50k", PATTERN_GPT2)
    data = textgen.mixed_c2(1 << 20, 1002).encode()
    assert tok.encode(data).tolist() == encode(data, v, PATTERN_GPT2)


def test_encode_session_1m_chars_100k_merges(pkg):
    v, tok = pair(pkg, "cl100k_session_100k", PATTERN_CL100K)
    data = textgen.agentic_session(1_000_000, 1003).encode()
    assert tok.encode(data).tolist() == encode(data, v, PATTERN_CL100K)


# --- batch ---------------------------------------------------------------

def test_token_offsets_match_oracle(pkg):
    # the device's token byte offsets against the oracle's definition
    for name, pat, data in (("gpt2_code_1k", PATTERN_GPT2, textgen.code_ascii(16384, 1001).encode()),
                            ("cl100k_session_100k", PATTERN_CL100K, textgen.agentic_session(200_000, 1003).encode()),
                            ("cl100k_session_100k", PATTERN_CL100K, textgen.adversarial(1 << 20, 1005, 0.02).encode())):
        v, tok = pair(pkg, name, pat)
        ids, offs = tok.encode_with_offsets(data)
        want_ids, want_offs = encode_with_offsets(data, v, pat)
        assert ids.tolist() == want_ids
        assert offs.tolist() == want_offs


def test_token_offsets_device_entry(pkg):
    import torch
    v, tok = pair(pkg, "cl100k_session_100k", PATTERN_CL100K)
    data = textgen.agentic_session(50_000, 1013).encode()
    n = len(data)
    d_text = torch.frombuffer(bytearray(data), dtype=torch.uint8).cuda()
    d_ids = torch.empty(n, dtype=torch.int32, device="cuda")
    d_off = torch.empty(n, dtype=torch.int64, device="cuda")
    d_st = torch.zeros(4, dtype=torch.int64, device="cuda")
    tok.encode_offsets_device(d_text.data_ptr(), n, d_ids.data_ptr(), d_off.data_ptr(), n, d_st.data_ptr(),
                              torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    st = d_st.cpu().tolist()
    assert st[0] == 0
    want_ids, want_offs = encode_with_offsets(data, v, PATTERN_CL100K)
    assert d_ids[:st[1]].cpu().tolist() == want_ids
    assert d_off[:st[1]].cpu().tolist() == want_offs


def test_pinned_host_buffers(pkg):
    # pinned buffers take the direct path (the boundary kernel reads the text
    # in place; the device writes ids, offsets and status into host memory);
    # same results as the oracle
    import ctypes
    import torch
    v, tok = pair(pkg, "cl100k_session_100k", PATTERN_CL100K)
    L = pkg.lib()
    # a pinned input is read in place by the boundary kernel: also runs that
    # reach past a chunk's halo (their edge states read the host buffer) and a
    # length that ends inside a chunk
    runs = _runs_at_chunk_edges([b"\r\n", b"7", b" "], [13, 17, 40], range(-2, 19, 4))[:150_001]
    # letter runs of many ids: one that the emit kernel stages with the rest
    # of its 512-byte chunk, and one in the next chunk, which then has more
    # ids than it stages
    rng = random.Random(1029)
    letters = bytes(rng.choice(b"abcdefghijklmnopqrstuvwxyz") for _ in range(4200))
    long_runs = b"x " + letters[:200] + b" " + b"ab " * 120 + letters[200:] + b" tail"
    for data in (textgen.agentic_session(100_000, 1021).encode(), b"x", b"  \r\n\t 12345 abc", runs, long_runs):
        n = len(data)
        h_text = torch.frombuffer(bytearray(data), dtype=torch.uint8).pin_memory()
        h_ids = torch.empty(n, dtype=torch.int32).pin_memory()
        h_off = torch.empty(n, dtype=torch.int64).pin_memory()
        got = ctypes.c_uint64()
        tp = ctypes.cast(h_text.data_ptr(), ctypes.POINTER(ctypes.c_uint8))
        ip = ctypes.cast(h_ids.data_ptr(), ctypes.POINTER(ctypes.c_int32))
        op = ctypes.cast(h_off.data_ptr(), ctypes.POINTER(ctypes.c_int64))
        assert L.tok_encode(tok._h, tp, n, ip, n, ctypes.byref(got)) == 0
        want_ids, want_offs = encode_with_offsets(data, v, PATTERN_CL100K)
        assert h_ids[:got.value].tolist() == want_ids
        assert L.tok_encode_offsets(tok._h, tp, n, ip, op, n, ctypes.byref(got)) == 0
        assert h_ids[:got.value].tolist() == want_ids and h_off[:got.value].tolist() == want_offs
    bad = b"abc " * 1000 + b"\xf0\x28\x8c\x28" + b" tail"
    h_text = torch.frombuffer(bytearray(bad), dtype=torch.uint8).pin_memory()
    h_ids = torch.empty(len(bad), dtype=torch.int32).pin_memory()
    got = ctypes.c_uint64()
    rc = L.tok_encode(tok._h, ctypes.cast(h_text.data_ptr(), ctypes.POINTER(ctypes.c_uint8)), len(bad),
                      ctypes.cast(h_ids.data_ptr(), ctypes.POINTER(ctypes.c_int32)), len(bad), ctypes.byref(got))
    with pytest.raises(Utf8Error) as e:
        encode(bad, v, PATTERN_CL100K)
    assert rc == pkg.TOK_EUTF8 and L.tok_error_offset(tok._h) == e.value.offset


def test_repair_append_matches_full_encoding(pkg):
    # session repair (Section 3.3): appends of agent-session text, of text that
    # extends the old text's last run (letters, digits, whitespace, CR/LF),
    # and to an old text without any cut
    rng = random.Random(17)
    for name, pat in (("cl100k_session_100k", PATTERN_CL100K), ("gpt2_session_100k", PATTERN_GPT2)):
        v, tok = pair(pkg, name, pat)
        s = textgen.agentic_session(400_000, 1031).encode()
        cases = []
        for _ in range(6):
            a = rng.randrange(1000, len(s) - 5000)
            cases.append((s[:a], s[a:a + rng.randrange(1, 3000)]))
        cases += [(b"the pipe", b"line"), (b"x = 12345", b"678 + 9"), (b"end  ", b"  \r\n\r\nmore"),
                  (b"abc", b"def"), ("caf\u00e9".encode(), "\u0301s".encode()), (b"", b"fresh start")]
        for old, delta in cases:
            try:
                old.decode("utf-8"), delta.decode("utf-8")
            except UnicodeDecodeError:
                continue
            oi, oo = tok.encode_with_offsets(old)
            ids, offs, re = tok.repair_append(old, oi, oo, delta)
            want = encode_with_offsets(old + delta, v, pat)
            assert (ids.tolist(), offs.tolist()) == want, (old[-20:], delta[:20])
            o_ids, o_offs, o_re = oracle_repair_append(old, oi.tolist(), oo.tolist(), delta, v, pat)
            assert re == o_re


def test_encode_batch_64_sessions(pkg, oracle_pool):
    # the 64-session batch in one tok_encode_batch call: every item's ids
    # against the oracle's
    v, tok = pair(pkg, "cl100k_session_100k", PATTERN_CL100K)
    items = [s.encode() for s in textgen.session_batch(64, 1004)]
    ids, off = tok.encode_batch(items)
    assert off[0] == 0 and off[-1] == len(ids) and np.all(np.diff(off) >= 0)
    want = oracle_pool.encode_many(items, os.path.join(VOC, "cl100k_session_100k.merges"), PATTERN_CL100K)
    for k, it in enumerate(items):
        assert ids[off[k]:off[k + 1]].tolist() == want[k][0], k
    # batch == singles
    for k in (0, 17, 63):
        assert tok.encode(items[k]).tolist() == ids[off[k]:off[k + 1]].tolist()


# --- adversarial ---------------------------------------------------------

@pytest.mark.parametrize("name,pattern", [("gpt2_session_100k", PATTERN_GPT2),
                                          ("cl100k_session_100k", PATTERN_CL100K)])
def test_adversarial_scaled_exact(pkg, name, pattern):
    v, tok = pair(pkg, name, pattern)
    data = textgen.adversarial(400_000, 1005, scale=0.02).encode()
    assert tok.encode(data).tolist() == encode(data, v, pattern)
    pieces = [p.encode() for p in textgen.adversarial_pieces(1005, scale=0.02)]
    ids, off = tok.encode_batch(pieces)
    for k, p in enumerate(pieces):
        assert ids[off[k]:off[k + 1]].tolist() == encode(p, v, pattern), k


@pytest.mark.parametrize("name,pattern", [("gpt2_session_100k", PATTERN_GPT2),
                                          ("cl100k_session_100k", PATTERN_CL100K)])
def test_adversarial_8mib_exact(pkg, oracle_pool, name, pattern):
    # the whole 8 MiB adversarial text: every fragment start of the
    # pre-tokenizer and every id, against the oracle
    v, tok = pair(pkg, name, pattern)
    data = textgen.adversarial(8 << 20, 1005).encode()
    want_ids, want_starts = oracle_pool.encode_long(data, os.path.join(VOC, name + ".merges"), pattern)
    starts = tok.pretokenize(data).tolist()
    assert len(starts) == len(want_starts)
    assert starts == want_starts
    ids = tok.encode(data).tolist()
    assert len(ids) == len(want_ids)
    assert ids == want_ids


# --- edge cases ------------------------------------------------------------

def test_empty_and_tiny(pkg):
    v, tok = pair(pkg, "cl100k_session_100k", PATTERN_CL100K)
    assert tok.encode(b"").tolist() == []
    # the Python-list output mode: the same ids as plain ints
    d = textgen.agentic_session(20_000, 1061).encode()
    lst = tok.encode_list(d)
    assert type(lst) is list and all(type(x) is int for x in lst[:10]) and lst == encode(d, v, PATTERN_CL100K)
    assert tok.encode_list(b"") == []
    for b in range(128):
        d = bytes([b])
        assert tok.encode(d).tolist() == encode(d, v, PATTERN_CL100K)
    ids, off = tok.encode_batch([b"", b"a", b"", b" ", b""])
    assert off.tolist() == [0, 0, 1, 1, 2, 2]


@pytest.mark.parametrize("pattern", [PATTERN_GPT2, PATTERN_CL100K])
def test_ragged_sizes_and_tier_edges(pkg, pattern):
    name = "gpt2_session_100k" if pattern == PATTERN_GPT2 else "cl100k_session_100k"
    v, tok = pair(pkg, name, pattern)
    base = textgen.agentic_session_bytes(20000, 77).encode()
    for n in (1, 15, 16, 17, 255, 256, 257, 1023, 1024, 1025, 4095, 4096, 4097, 8191, 8193, 12289):
        d = base[:n]
        while d and (d[-1] & 0xC0) == 0x80:
            d = d[:-1]
        assert tok.encode(d).tolist() == encode(d, v, pattern), n
    rnd = random.Random(5)
    for n in (16, 17, 255, 256, 257, 300, 1000, 5000, 20000):
        for alpha in ("abcdefghij", "0123456789", "=", " ", "ab"):
            d = ("x " + "".join(rnd.choice(alpha) for _ in range(n)) + " y").encode()
            assert tok.encode(d).tolist() == encode(d, v, pattern), (n, alpha)


@pytest.mark.parametrize("pattern", [PATTERN_GPT2, PATTERN_CL100K])
def test_warp_engine_tiers(pkg, pattern):
    # fragments around the warp engines' limits: a batch whose fragments are
    # all at most 16 bytes merges step by step, one with a longer fragment
    # (up to 32) in certified sweeps, longer fragments go to the CTA engines;
    # rare letters keep the fragments from being whole tokens
    name = "gpt2_session_100k" if pattern == PATTERN_GPT2 else "cl100k_session_100k"
    v, tok = pair(pkg, name, pattern)
    rnd = random.Random(11)
    for lens in ((2, 8, 15, 16), (16, 17), (15, 16, 17, 18), (24, 31, 32), (31, 32, 33, 34), (2, 3, 16, 32, 40)):
        words = [" " + "".join(rnd.choice("qzxjkvwy") for _ in range(rnd.choice(lens) - 1)) for _ in range(300)]
        d = "".join(words).encode()
        assert tok.encode(d).tolist() == encode(d, v, pattern), lens


def test_invalid_utf8_offsets(pkg):
    _, tok = pair(pkg, "cl100k_session_100k", PATTERN_CL100K)
    cases = [b"abc\xe4\xb8", b"\x80abc", b"ab\xc0\xafcd", b"x\xed\xa0\x80y", b"\xf4\x90\x80\x80", b"ok \xff",
             b"a" * 5000 + b"\xe2\x82", b"a" * 4094 + b"\xe4\xb8\xad\x80" + b"b" * 10]
    for d in cases:
        with pytest.raises(Utf8Error) as ref:
            encode(d, Vocab.from_merges([]), 0)
        with pytest.raises(pkg.TokError) as e:
            tok.encode(d)
        assert e.value.code == pkg.TOK_EUTF8 and e.value.offset == ref.value.offset, d[:20]
    # batch items are validated on their own: a sequence may not span items
    with pytest.raises(pkg.TokError) as e:
        tok.encode_batch([b"ab\xe4\xb8", b"\xadcd"])
    assert e.value.code == pkg.TOK_EUTF8 and e.value.offset == 2


def test_non_monotone_vocabulary_falls_back_exactly(pkg):
    # "abc" is made by (ab,c) at rank 1 and again by (a,bc) at rank 4, after
    # (abc,d) used it at rank 2: merges can create lower-rank pairs
    toks = [bytes([b]) for b in range(256)] + [b"ab", b"abc", b"abcd", b"bc", b"cd", b"dd"]
    ix = {t: i for i, t in enumerate(toks)}
    merges = [(ix[b"a"], ix[b"b"]), (ix[b"ab"], ix[b"c"]), (ix[b"abc"], ix[b"d"]), (ix[b"b"], ix[b"c"]),
              (ix[b"a"], ix[b"bc"]), (ix[b"c"], ix[b"d"]), (ix[b"d"], ix[b"d"])]
    v = Vocab(toks, merges)
    assert not v.monotone()
    tok = pkg.Tokenizer(toks, merges, PATTERN_GPT2)
    rnd = random.Random(6)
    words = ["".join(rnd.choice("abcd") for _ in range(n)) for n in (3, 10, 16, 17, 40, 200, 256, 300, 2000)]
    data = " ".join(words).encode()
    assert tok.encode(data).tolist() == encode(data, v, PATTERN_GPT2)


def test_device_entry_points(pkg):
    import torch
    v, tok = pair(pkg, "cl100k_session_100k", PATTERN_CL100K)
    data = textgen.agentic_session(200_000, 11).encode()
    want = tok.encode(data)
    d_text = torch.frombuffer(bytearray(data), dtype=torch.uint8).cuda()
    d_ids = torch.empty(len(data), dtype=torch.int32, device="cuda")
    d_st = torch.zeros(4, dtype=torch.int64, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    tok.encode_device(d_text.data_ptr(), len(data), d_ids.data_ptr(), len(data), d_st.data_ptr(), stream)
    torch.cuda.synchronize()
    st = d_st.cpu().tolist()
    assert st[0] == 0 and st[2] == -1
    assert d_ids[:st[1]].cpu().numpy().tolist() == want.tolist()
    # batch on the device
    items = [data[:5000], data[5000:5000], data[5000:70001], data[70001:]]
    items = [it for it in items]
    starts = np.cumsum([0] + [len(x) for x in items]).astype(np.int64)
    d_items = torch.from_numpy(starts).cuda()
    d_off = torch.zeros(len(items) + 1, dtype=torch.int64, device="cuda")
    tok.encode_batch_device(d_text.data_ptr(), len(data), d_items.data_ptr(), len(items), d_ids.data_ptr(),
                            len(data), d_off.data_ptr(), d_st.data_ptr(), stream)
    torch.cuda.synchronize()
    ids_h, off_h = tok.encode_batch(items)
    assert d_off.cpu().tolist() == off_h.tolist()
    assert d_ids[:int(off_h[-1])].cpu().numpy().tolist() == ids_h.tolist()


def test_device_status_whatever_it_held_before(pkg):
    # the caller's status buffer holds garbage, then an earlier call's error:
    # after each call it holds exactly this call's result (the boundary
    # kernel sets the code, the emit kernel's last chunk completes the rest)
    import torch
    from oracle.utf8 import decode_utf8
    v, tok = pair(pkg, "cl100k_session_100k", PATTERN_CL100K)
    stream = torch.cuda.current_stream().cuda_stream
    good = textgen.agentic_session(120_000, 21).encode()
    small = textgen.agentic_session(3_000, 22).encode()
    bad = good[:70_001] + b"\xff" + good[70_001:]
    with pytest.raises(Utf8Error) as e:
        decode_utf8(bad)
    bad_at = e.value.offset
    n = len(bad)
    d_text = torch.empty(n, dtype=torch.uint8, device="cuda")
    d_ids = torch.empty(n, dtype=torch.int32, device="cuda")
    d_st = torch.tensor([-77, 123456789, 42, 99], dtype=torch.int64, device="cuda")

    def put(data):
        if data:
            d_text[:len(data)] = torch.frombuffer(bytearray(data), dtype=torch.uint8).cuda()

    def run(data):
        put(data)
        tok.encode_device(d_text.data_ptr(), len(data), d_ids.data_ptr(), n, d_st.data_ptr(), stream)
        torch.cuda.synchronize()
        return d_st.cpu().tolist()

    for data in (good, small):
        d_st.copy_(torch.tensor([-77, 123456789, 42, 99]))
        want = encode(data, v, PATTERN_CL100K)
        assert run(data) == [pkg.TOK_OK, len(want), -1, 0]
        assert d_ids[:len(want)].cpu().tolist() == want
    st = run(bad)
    assert st[0] == pkg.TOK_EUTF8 and st[2] == bad_at
    assert run(good) == [pkg.TOK_OK, len(encode(good, v, PATTERN_CL100K)), -1, 0]
    st = run(bad)
    assert st[0] == pkg.TOK_EUTF8 and st[2] == bad_at
    assert run(b"") == [pkg.TOK_OK, 0, -1, 0]
    # a batch after an error, its status buffer full of garbage
    items = [good[:40_000], b"", good[40_000:]]
    starts = torch.tensor(np.cumsum([0] + [len(x) for x in items]).astype(np.int64)).cuda()
    d_off = torch.full((len(items) + 1,), -5, dtype=torch.int64, device="cuda")
    run(bad)
    put(good)
    d_st.copy_(torch.tensor([-77, 123456789, 42, 99]))
    tok.encode_batch_device(d_text.data_ptr(), len(good), starts.data_ptr(), len(items), d_ids.data_ptr(), n,
                            d_off.data_ptr(), d_st.data_ptr(), stream)
    torch.cuda.synchronize()
    ids_h, off_h = tok.encode_batch(items)
    assert d_st.cpu().tolist() == [pkg.TOK_OK, int(off_h[-1]), -1, 0]
    assert d_off.cpu().tolist() == off_h.tolist()


# --- o200k-style pattern --------------------------------------------------------

def test_o200k_style_encode_matches_oracle(pkg, oracle_pool):
    # the o200k-style pattern (this library's own definition) with the
    # 100k-merge session vocabulary: the 1M-character session, code with
    # paths and camelCase, the scaled adversarial text and a batch
    path = os.path.join(VOC, "cl100k_session_100k.merges")
    v = Vocab.load_merges(path)
    tok = pkg.Tokenizer.from_merges_file(path, PATTERN_O200K)
    session = textgen.agentic_session(1_000_000, 1003).encode()
    want_ids, want_starts = oracle_pool.encode_long(session, path, PATTERN_O200K)
    assert tok.pretokenize(session).tolist() == want_starts
    assert tok.encode(session).tolist() == want_ids
    code = textgen.code_ascii(300_000, 1051).encode()
    assert tok.encode(code).tolist() == encode(code, v, PATTERN_O200K)
    adv = textgen.adversarial(400_000, 1005, scale=0.02).encode()
    ids, offs = tok.encode_with_offsets(adv)
    assert (ids.tolist(), offs.tolist()) == encode_with_offsets(adv, v, PATTERN_O200K)
    items = [x.encode() for x in textgen.session_batch(8, 1052, hi=1 << 16)]
    ids, off = tok.encode_batch(items)
    for k, it in enumerate(items):
        assert ids[off[k]:off[k + 1]].tolist() == encode(it, v, PATTERN_O200K), k
    # repair after appends
    old, delta = session[:30_000], session[30_000:31_500]
    oi, oo = tok.encode_with_offsets(old)
    got = tok.repair_append(old, oi, oo, delta)
    assert (got[0].tolist(), got[1].tolist()) == encode_with_offsets(old + delta, v, PATTERN_O200K)
    tok.close()


# --- ignore_merges -------------------------------------------------------------

def test_deepseek_style_encode_matches_oracle(pkg, oracle_pool):
    # the DeepSeek-style pattern (this library's own definition) with the
    # 100k-merge session vocabulary: the 1M-character session, the mixed text
    # with 10% CJK, Japanese and Korean runs among Latin words, the scaled
    # adversarial text with offsets, a batch
    path = os.path.join(VOC, "cl100k_session_100k.merges")
    v = Vocab.load_merges(path)
    tok = pkg.Tokenizer.from_merges_file(path, PATTERN_DEEPSEEK)
    session = textgen.agentic_session(1_000_000, 1003).encode()
    want_ids, want_starts = oracle_pool.encode_long(session, path, PATTERN_DEEPSEEK)
    assert tok.pretokenize(session).tolist() == want_starts
    assert tok.encode(session).tolist() == want_ids
    mixed = textgen.mixed_c2(300_000, 1061).encode()
    assert tok.pretokenize(mixed).tolist() == oracle_starts(mixed, PATTERN_DEEPSEEK)
    assert tok.encode(mixed).tolist() == encode(mixed, v, PATTERN_DEEPSEEK)
    rnd = random.Random(1062)
    words = ["カーテン", "ひらがな", "한국어", "漢字", "々", "〆切", "text", "naïve", " ", "  ", ".", ",", "'s", "1234",
             "\n", "\r\n", "Ωmega", "ㄅ", "ｱｲｳ", "𠀀"]
    cjk = "".join(rnd.choice(words) for _ in range(40_000)).encode()
    assert tok.pretokenize(cjk).tolist() == oracle_starts(cjk, PATTERN_DEEPSEEK)
    assert tok.encode(cjk).tolist() == encode(cjk, v, PATTERN_DEEPSEEK)
    adv = textgen.adversarial(400_000, 1005, scale=0.02).encode()
    ids, offs = tok.encode_with_offsets(adv)
    assert (ids.tolist(), offs.tolist()) == encode_with_offsets(adv, v, PATTERN_DEEPSEEK)
    items = [x.encode() for x in textgen.session_batch(8, 1063, hi=1 << 16)]
    ids, off = tok.encode_batch(items)
    for k, it in enumerate(items):
        assert ids[off[k]:off[k + 1]].tolist() == encode(it, v, PATTERN_DEEPSEEK), k
    tok.close()


def test_ignore_merges_matches_oracle(pkg):
    # a vocabulary with tokens that do not encode to themselves: with the flag
    # a fragment that is such a token is that token (Section 4.2), every other
    # fragment is BPE; the session vocabulary on session text and on a long
    # letter run (no split into pieces under the flag)
    toks = [bytes([b]) for b in range(256)] + [b"ab", b"bc", b"abc", b" ab", b" abc"]
    ix = {t: i for i, t in enumerate(toks)}
    merges = [(ix[b"a"], ix[b"b"]), (ix[b"b"], ix[b"c"]), (ix[b"a"], ix[b"bc"]), (ix[b" "], ix[b"ab"]),
              (ix[b" "], ix[b"abc"])]
    v = Vocab(toks, merges)
    data = b"abc abc abcc xabc  abc bcabc " * 50
    for pat in (PATTERN_GPT2, PATTERN_CL100K):
        tok = pkg.Tokenizer(toks, merges, pat, ignore_merges=True)
        assert tok.encode(data).tolist() == encode(data, v, pat, ignore_merges=True)
        assert encode(data, v, pat, ignore_merges=True) != encode(data, v, pat)
        tok.close()
    path = os.path.join(VOC, "cl100k_session_100k.merges")
    vs = Vocab.load_merges(path)
    tok = pkg.Tokenizer.from_merges_file(path, PATTERN_CL100K, ignore_merges=True)
    for d in (textgen.agentic_session(200_000, 1041).encode(), textgen.adversarial(600_000, 1005, scale=0.03).encode()):
        ids, offs = tok.encode_with_offsets(d)
        want = encode_with_offsets(d, vs, PATTERN_CL100K, ignore_merges=True)
        assert (ids.tolist(), offs.tolist()) == want
    items = [s.encode() for s in textgen.session_batch(6, 1042, hi=1 << 16)]
    ids, off = tok.encode_batch(items)
    for k, it in enumerate(items):
        assert ids[off[k]:off[k + 1]].tolist() == encode(it, vs, PATTERN_CL100K, ignore_merges=True)
    tok.close()
