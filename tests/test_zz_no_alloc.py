"""tok_pretokenize_device_noalloc: the pre-tokenizer for callers that cannot
allocate device memory (for example code running inside another framework's
memory pool, or under a fixed memory budget).  It keeps its scratch in a
fixed array inside the library, so the test checks that two calls in a row,
each reusing that array, give exactly the fragment starts of the allocating
entry point (tok_pretokenize), and that errors are reported the same way.

Collected last on purpose: a failure here never hides another test."""
import ctypes

import numpy as np
import pytest

import textgen

pytestmark = pytest.mark.gpu


def _starts_from_bits(words, n):
    bits = np.unpackbits(words.view(np.uint8), bitorder="little")[:n]
    return np.nonzero(bits)[0].tolist()


def test_noalloc_pretokenizer_matches_allocating_entry_point():
    import torch

    from exact_bpe_tokenization_utf_gb300 import _build
    _build.build()
    import exact_bpe_tokenization_utf_gb300 as pkg
    L = pkg.lib()
    stream = torch.cuda.current_stream().cuda_stream
    for pattern in (pkg.PATTERN_GPT2, pkg.PATTERN_CL100K):
        tok = pkg.Tokenizer.from_merges([], pattern)
        texts = [textgen.agentic_session(300_000, 50 + pattern).encode(),
                 textgen.adversarial(200_003, 60 + pattern, scale=0.02).encode()]
        for data in texts:  # two calls in a row share the scratch array
            n = len(data)
            words = -(-n // 32)
            d_text = torch.frombuffer(bytearray(data), dtype=torch.uint8).cuda()
            d_bits = torch.full((words,), -1, dtype=torch.int32, device="cuda")
            d_st = torch.full((2,), 7, dtype=torch.int64, device="cuda")
            rc = L.tok_pretokenize_device_noalloc(pattern, d_text.data_ptr(), n, d_bits.data_ptr(),
                                                  d_st.data_ptr(), ctypes.c_void_p(stream))
            torch.cuda.synchronize()
            assert rc == pkg.TOK_OK
            assert d_st.cpu().tolist() == [pkg.TOK_OK, -1]
            got = _starts_from_bits(d_bits.cpu().numpy(), n)
            assert got == tok.pretokenize(data).tolist()
        # malformed input: same error offset as the allocating entry point
        bad = b"a" * 5000 + b"\xe4\xb8" + b"b" * 10
        d_text = torch.frombuffer(bytearray(bad), dtype=torch.uint8).cuda()
        d_bits = torch.zeros(-(-len(bad) // 32), dtype=torch.int32, device="cuda")
        d_st = torch.zeros(2, dtype=torch.int64, device="cuda")
        rc = L.tok_pretokenize_device_noalloc(pattern, d_text.data_ptr(), len(bad), d_bits.data_ptr(),
                                              d_st.data_ptr(), ctypes.c_void_p(stream))
        torch.cuda.synchronize()
        with pytest.raises(pkg.TokError) as e:
            tok.pretokenize(bad)
        assert rc == pkg.TOK_OK and d_st.cpu().tolist() == [pkg.TOK_EUTF8, e.value.offset]
        # invalid arguments are rejected before touching the device
        assert L.tok_pretokenize_device_noalloc(pattern, d_text.data_ptr(), len(bad), d_bits.data_ptr(),
                                                None, ctypes.c_void_p(stream)) == pkg.TOK_EINVAL
        assert L.tok_pretokenize_device_noalloc(7, d_text.data_ptr(), len(bad), d_bits.data_ptr(),
                                                d_st.data_ptr(), ctypes.c_void_p(stream)) == pkg.TOK_EINVAL
        tok.close()
