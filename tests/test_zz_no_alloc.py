"""tok_pretokenize_device_noalloc: the pre-tokenizer for callers that cannot
allocate device memory (code that runs inside another framework's memory pool
or arena, code that must not cause the device-wide synchronisation a
cudaMalloc or cudaFree can bring, hosts held to a fixed memory budget).  It
keeps its scratch in a fixed array inside the library, so the test runs two
calls in a row, each reusing that array, and checks each against the oracle's
fragment starts and against the allocating entry point (tok_pretokenize);
errors, the padding bits of the last bitmask word, the empty text and the
length bound are checked too.

Collected last on purpose: a failure here never hides another test."""
import ctypes

import numpy as np
import pytest

import textgen
from oracle.encode import pretoken_byte_spans
from oracle.utf8 import Utf8Error, decode_utf8

pytestmark = pytest.mark.gpu


def _bits(words, n):
    return np.unpackbits(np.ascontiguousarray(words).view(np.uint8), bitorder="little")[:n]


def _oracle_starts(data, pattern):
    return [a for a, _ in pretoken_byte_spans(data, pattern)]


def _call(L, pattern, d_text, n, d_bits, d_st, stream):
    return L.tok_pretokenize_device_noalloc(pattern, d_text, n, d_bits, d_st, ctypes.c_void_p(stream))


def test_noalloc_pretokenizer_matches_oracle():
    import torch

    from exact_bpe_tokenization_utf_gb300 import _build
    _build.build()
    import exact_bpe_tokenization_utf_gb300 as pkg
    L = pkg.lib()
    stream = torch.cuda.current_stream().cuda_stream
    for pattern in (pkg.PATTERN_GPT2, pkg.PATTERN_CL100K, pkg.PATTERN_O200K, pkg.PATTERN_DEEPSEEK):
        tok = pkg.Tokenizer.from_merges([], pattern)
        # lengths that end inside a bitmask word (n % 32 != 0) and inside a chunk
        texts = [textgen.agentic_session(300_000, 50 + pattern).encode(),
                 textgen.adversarial(200_003, 60 + pattern, scale=0.02).encode()]
        for data in texts:  # two calls in a row share the scratch array
            n = len(data)
            words = -(-n // 32)
            d_text = torch.frombuffer(bytearray(data), dtype=torch.uint8).cuda()
            d_bits = torch.full((words + 4,), -1, dtype=torch.int32, device="cuda")
            d_st = torch.full((2,), 7, dtype=torch.int64, device="cuda")
            rc = _call(L, pattern, d_text.data_ptr(), n, d_bits.data_ptr(), d_st.data_ptr(), stream)
            torch.cuda.synchronize()
            assert rc == pkg.TOK_OK
            assert d_st.cpu().tolist() == [pkg.TOK_OK, -1]
            h = d_bits.cpu().numpy()
            got = np.nonzero(_bits(h[:words], n))[0].tolist()
            assert got == _oracle_starts(data, pattern)
            assert got == tok.pretokenize(data).tolist()
            # bits at p >= n in the last word are 0; words past it untouched
            if n % 32:
                assert int(h[words - 1]) & ((0xFFFFFFFF << (n % 32)) & 0xFFFFFFFF) == 0
            assert h[words:].tolist() == [-1] * 4
        # malformed input: the oracle's offset of the first bad byte
        bad = b"a" * 5000 + b"\xe4\xb8" + b"b" * 10
        with pytest.raises(Utf8Error) as ref:
            decode_utf8(bad)
        d_text = torch.frombuffer(bytearray(bad), dtype=torch.uint8).cuda()
        d_bits = torch.zeros(-(-len(bad) // 32), dtype=torch.int32, device="cuda")
        d_st = torch.zeros(2, dtype=torch.int64, device="cuda")
        rc = _call(L, pattern, d_text.data_ptr(), len(bad), d_bits.data_ptr(), d_st.data_ptr(), stream)
        torch.cuda.synchronize()
        assert rc == pkg.TOK_OK and d_st.cpu().tolist() == [pkg.TOK_EUTF8, ref.value.offset]
        # the next well-formed call reports no error although the scratch
        # still holds the previous call's error word
        good = b"fine text 123"
        d_good = torch.frombuffer(bytearray(good), dtype=torch.uint8).cuda()
        rc = _call(L, pattern, d_good.data_ptr(), len(good), d_bits.data_ptr(), d_st.data_ptr(), stream)
        torch.cuda.synchronize()
        assert rc == pkg.TOK_OK and d_st.cpu().tolist() == [pkg.TOK_OK, -1]
        # an empty text writes only the status (no host sync, no bitmask)
        d_st.fill_(7)
        rc = _call(L, pattern, None, 0, None, d_st.data_ptr(), stream)
        torch.cuda.synchronize()
        assert rc == pkg.TOK_OK and d_st.cpu().tolist() == [pkg.TOK_OK, -1]
        # refused on the host before anything is enqueued: NULL status, an
        # unknown pattern, a length beyond 2^34 - 2
        d_st.fill_(7)
        assert _call(L, pattern, d_text.data_ptr(), len(bad), d_bits.data_ptr(), None, stream) == pkg.TOK_EINVAL
        assert _call(L, 7, d_text.data_ptr(), len(bad), d_bits.data_ptr(), d_st.data_ptr(), stream) == pkg.TOK_EINVAL
        assert _call(L, pattern, d_text.data_ptr(), (1 << 34) - 1, d_bits.data_ptr(), d_st.data_ptr(),
                     stream) == pkg.TOK_EINVAL
        torch.cuda.synchronize()
        assert d_st.cpu().tolist() == [7, 7]
        tok.close()
