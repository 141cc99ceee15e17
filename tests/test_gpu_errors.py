"""Error paths of the C ABI, every failure made on the host: allocation
failures injected with tok_debug_fail_alloc (TOK_ENOMEM, the handle usable
afterwards, no device memory kept), output buffers that are too small
(TOK_EBUF with the required size), and arguments that do not fit (TOK_EINVAL:
old token offsets that do not belong to the text, an old length beyond the
text, NULL pointers).  Nothing here faults or stalls the GPU."""
import ctypes
import os

import numpy as np
import pytest

import textgen
from oracle.encode import encode, encode_with_offsets
from oracle.pretokenize import PATTERN_CL100K
from oracle.vocab import Vocab

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
VOCAB = os.path.join(ROOT, "data", "vocabs", "cl100k_session_100k.merges")

U8P, I32P, I64P, U64P = (ctypes.POINTER(ctypes.c_uint8), ctypes.POINTER(ctypes.c_int32),
                         ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_uint64))


@pytest.fixture(scope="module")
def env():
    from exact_bpe_tokenization_utf_gb300 import _build
    _build.build()
    import exact_bpe_tokenization_utf_gb300 as pkg
    tok = pkg.Tokenizer.from_merges_file(VOCAB, pkg.PATTERN_CL100K)
    yield pkg, tok, Vocab.load_merges(VOCAB)
    tok.close()


def _p(a, t):
    return a.ctypes.data_as(t)


def _encode_raw(L, h, data, cap):
    """tok_encode into a pageable buffer of capacity cap: (rc, *n_ids, ids)."""
    src = np.frombuffer(data, dtype=np.uint8) if data else np.zeros(1, np.uint8)
    ids = np.full(max(cap, 1), -7, dtype=np.int32)
    n = ctypes.c_uint64(12345)
    rc = L.tok_encode(h, _p(src, U8P), len(data), _p(ids, I32P), cap, ctypes.byref(n))
    return rc, n.value, ids


def _free_bytes():
    import torch
    torch.cuda.synchronize()
    return torch.cuda.mem_get_info()[0]


def _fail_each_allocation(pkg, L, tok, data):
    """Arm the hook at the 1st, 2nd, ... allocation of tok's next call on
    data until the call gets through; returns (failures, ids)."""
    k = 1
    while True:
        assert L.tok_debug_fail_alloc(tok._h, k) == pkg.TOK_OK
        try:
            ids = tok.encode(data)
        except pkg.TokError as e:
            assert e.code == pkg.TOK_ENOMEM, str(e)
            assert b"allocation failed" in L.tok_last_error(tok._h)
            k += 1
            continue
        L.tok_debug_fail_alloc(tok._h, 0)
        return k - 1, ids


def test_out_of_memory_is_reported_and_the_handle_recovers(env):
    pkg, tok, v = env
    L = pkg.lib()
    small = textgen.agentic_session(20_000, 71).encode()
    big = textgen.agentic_session(2_000_000, 72).encode()
    bigger = textgen.agentic_session(3_000_000, 73).encode()
    want = encode(big, v, PATTERN_CL100K)
    tok2 = pkg.Tokenizer.from_merges_file(VOCAB, pkg.PATTERN_CL100K)
    try:
        assert tok2.encode(small).tolist() == encode(small, v, PATTERN_CL100K)
        # every allocation of the workspace growth in turn: the call fails
        # with TOK_ENOMEM and frees what it had; then the call gets through
        fails, ids = _fail_each_allocation(pkg, L, tok2, big)
        assert fails >= 10
        assert ids.tolist() == want
        assert tok2.encode(small).tolist() == encode(small, v, PATTERN_CL100K)
        held = _free_bytes()
        # the same for a growth from the big workspace to a bigger one; back at
        # the big size the device holds what it held before: none of the
        # failed growths kept memory (tolerance: the driver's page granularity)
        fails2, _ = _fail_each_allocation(pkg, L, tok2, bigger)
        assert fails2 == fails
        tok2.close()
        tok2 = pkg.Tokenizer.from_merges_file(VOCAB, pkg.PATTERN_CL100K)
        assert tok2.encode(big).tolist() == want
        assert abs(_free_bytes() - held) < (16 << 20)
    finally:
        if tok2._h:
            L.tok_debug_fail_alloc(tok2._h, 0)
        tok2.close()


def test_out_of_memory_in_item_offset_and_pinned_buffers(env):
    pkg, tok, v = env
    L = pkg.lib()
    tok2 = pkg.Tokenizer.from_merges_file(VOCAB, pkg.PATTERN_CL100K)
    try:
        items = [b"first item", b"", b"third  item 123"]
        tok2.encode(b"x" * 4096)                 # workspace, so the batch's first allocation is its item buffers
        for k in (1, 2, 3):                      # device item starts, device item offsets, pinned host items
            L.tok_debug_fail_alloc(tok2._h, k)
            with pytest.raises(pkg.TokError) as e:
                tok2.encode_batch(items)
            assert e.value.code == pkg.TOK_ENOMEM
        L.tok_debug_fail_alloc(tok2._h, 0)
        ids, off = tok2.encode_batch(items)
        for j, it in enumerate(items):
            assert ids[off[j]:off[j + 1]].tolist() == encode(it, v, PATTERN_CL100K)
        # the token offset buffer, allocated on the first call that wants offsets
        data = textgen.agentic_session(5_000, 74).encode()
        L.tok_debug_fail_alloc(tok2._h, 1)
        with pytest.raises(pkg.TokError) as e:
            tok2.encode_with_offsets(data)
        assert e.value.code == pkg.TOK_ENOMEM
        L.tok_debug_fail_alloc(tok2._h, 0)
        got = tok2.encode_with_offsets(data)
        assert (got[0].tolist(), got[1].tolist()) == encode_with_offsets(data, v, PATTERN_CL100K)
        assert L.tok_debug_fail_alloc(None, 1) == pkg.TOK_EINVAL
    finally:
        tok2.close()


def test_output_too_small_reports_the_required_size(env):
    import torch
    pkg, tok, v = env
    L = pkg.lib()
    data = textgen.agentic_session(30_000, 75).encode()
    want = encode(data, v, PATTERN_CL100K)
    n = len(want)
    for cap in (0, 1, n - 1):
        rc, got_n, ids = _encode_raw(L, tok._h, data, cap)
        assert rc == pkg.TOK_EBUF and got_n == n
    rc, got_n, ids = _encode_raw(L, tok._h, data, n)       # exactly enough (cap < len: the copy path)
    assert rc == pkg.TOK_OK and got_n == n and ids[:n].tolist() == want
    # pinned output smaller than the text: the copy path, same contract
    h_ids = torch.empty(n, dtype=torch.int32).pin_memory()
    src = np.frombuffer(data, dtype=np.uint8)
    cnt = ctypes.c_uint64()
    ip = ctypes.cast(h_ids.data_ptr(), I32P)
    assert L.tok_encode(tok._h, _p(src, U8P), len(data), ip, n - 1, ctypes.byref(cnt)) == pkg.TOK_EBUF
    assert cnt.value == n
    assert L.tok_encode(tok._h, _p(src, U8P), len(data), ip, n, ctypes.byref(cnt)) == pkg.TOK_OK
    assert cnt.value == n and h_ids.tolist() == want
    # with offsets
    offs = np.zeros(n, dtype=np.int64)
    ids = np.zeros(n, dtype=np.int32)
    assert L.tok_encode_offsets(tok._h, _p(src, U8P), len(data), _p(ids, I32P), _p(offs, I64P), n - 1,
                                ctypes.byref(cnt)) == pkg.TOK_EBUF and cnt.value == n
    # batch: item_off[n] receives the required capacity
    items = [data[:10_000], data[10_000:10_000], data[10_000:]]
    total = sum(len(encode(it, v, PATTERN_CL100K)) for it in items)
    arrs = [np.frombuffer(x, dtype=np.uint8) if x else np.zeros(1, np.uint8) for x in items]
    ptrs = (U8P * 3)(*[_p(a, U8P) for a in arrs])
    lens = np.array([len(x) for x in items], dtype=np.uint64)
    item_off = np.zeros(4, dtype=np.uint64)
    ids = np.zeros(total, dtype=np.int32)
    assert L.tok_encode_batch(tok._h, ptrs, _p(lens, U64P), 3, _p(ids, I32P), total - 1,
                              _p(item_off, U64P)) == pkg.TOK_EBUF
    assert int(item_off[3]) == total
    assert L.tok_encode_batch(tok._h, ptrs, _p(lens, U64P), 3, _p(ids, I32P), total,
                              _p(item_off, U64P)) == pkg.TOK_OK
    assert int(item_off[3]) == total
    # device entry points need cap >= len, checked before any launch
    d_text = torch.frombuffer(bytearray(data), dtype=torch.uint8).cuda()
    d_ids = torch.empty(len(data), dtype=torch.int32, device="cuda")
    d_st = torch.full((4,), 9, dtype=torch.int64, device="cuda")
    rc = L.tok_encode_device(tok._h, d_text.data_ptr(), len(data), d_ids.data_ptr(), len(data) - 1,
                             d_st.data_ptr(), None)
    torch.cuda.synchronize()
    assert rc == pkg.TOK_EBUF and d_st.cpu().tolist() == [9, 9, 9, 9]


def _repair_raw(L, h, old, delta, old_ids, old_offs, cap, old_len=None):
    text = old + delta
    src = np.frombuffer(text, dtype=np.uint8) if text else np.zeros(1, np.uint8)
    oi = np.ascontiguousarray(old_ids, dtype=np.int32)
    oo = np.ascontiguousarray(old_offs, dtype=np.int64)
    ids = np.zeros(max(cap, 1), dtype=np.int32)
    offs = np.zeros(max(cap, 1), dtype=np.int64)
    n, re = ctypes.c_uint64(), ctypes.c_uint64()
    rc = L.tok_repair_append(h, _p(src, U8P), len(old) if old_len is None else old_len, len(text), _p(oi, I32P),
                             _p(oo, I64P), len(oi), _p(ids, I32P), _p(offs, I64P), cap, ctypes.byref(n),
                             ctypes.byref(re))
    return rc, n.value, ids, offs


def test_repair_errors(env):
    pkg, tok, v = env
    L = pkg.lib()
    old = textgen.agentic_session(20_000, 76).encode()
    delta = b" appended text, and more of it 12345\n"
    oi, oo = tok.encode_with_offsets(old)
    want_ids, want_offs = encode_with_offsets(old + delta, v, PATTERN_CL100K)
    n = len(want_ids)
    rc, got, ids, offs = _repair_raw(L, tok._h, old, delta, oi, oo, n)
    assert rc == pkg.TOK_OK and got == n and ids[:n].tolist() == want_ids and offs[:n].tolist() == want_offs
    # too small: while the kept tokens fit, and when they alone do not
    for cap in (n - 1, len(oi) // 2, 0):
        rc, got, _, _ = _repair_raw(L, tok._h, old, delta, oi, oo, cap)
        assert rc == pkg.TOK_EBUF and got == n, cap
    # old offsets that do not belong to the text: shifted by one byte
    rc, _, _, _ = _repair_raw(L, tok._h, old, delta, oi, oo + 1, n)
    assert rc == pkg.TOK_EINVAL
    assert b"do not belong" in L.tok_last_error(tok._h)
    # an old length beyond the text, and a NULL output
    rc, _, _, _ = _repair_raw(L, tok._h, old, delta, oi, oo, n, old_len=len(old) + len(delta) + 1)
    assert rc == pkg.TOK_EINVAL
    src = np.frombuffer(old, dtype=np.uint8)
    cnt = ctypes.c_uint64()
    assert L.tok_repair_append(tok._h, _p(src, U8P), len(old), len(old), _p(oi, I32P), _p(oo, I64P), len(oi),
                               None, None, n, ctypes.byref(cnt), None) == pkg.TOK_EINVAL
    # the handle still encodes after the refusals
    assert tok.encode(old + delta).tolist() == want_ids
