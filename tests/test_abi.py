"""The C-ABI library builds, loads without a GPU, and exports every entry
point include/tok.h declares; the binding knows the same set."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    with open(os.path.join(ROOT, "include", "tok.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tok_[a-z_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def libpath():
    from exact_bpe_tokenization_utf_gb300 import _build
    return _build.build()


def test_library_exports_every_declared_symbol(libpath):
    syms = declared_symbols()
    assert len(syms) >= 12
    L = ctypes.CDLL(libpath)
    for s in syms:
        assert hasattr(L, s), s


def test_binding_symbol_list_matches_header():
    import exact_bpe_tokenization_utf_gb300 as pkg
    assert sorted(pkg.SYMBOLS) == declared_symbols()


def test_binding_loads_and_load_validates(libpath):
    # tok_load's validation runs on the host before any device call
    import exact_bpe_tokenization_utf_gb300 as pkg
    L = pkg.lib()
    h = ctypes.c_void_p()
    rc = L.tok_load(None, None, 0, None, 0, 0, ctypes.byref(h))
    assert rc == pkg.TOK_EINVAL
    with pytest.raises(pkg.TokError) as e:
        pkg.Tokenizer([bytes([b]) for b in range(255)], [], 0)
    assert e.value.code == pkg.TOK_EMERGES
    with pytest.raises(pkg.TokError) as e:
        pkg.Tokenizer([bytes([b]) for b in range(256)], [(97, 98)], 0)  # result "ab" missing
    assert e.value.code == pkg.TOK_EMERGES
    with pytest.raises(pkg.TokError) as e:
        pkg.Tokenizer([bytes([b]) for b in range(256)] + [b"aa"], [(97, 97), (97, 97)], 0)
    assert e.value.code == pkg.TOK_EMERGES
    with pytest.raises(pkg.TokError) as e:
        pkg.Tokenizer([bytes([b]) for b in range(256)], [], 7)
    assert e.value.code == pkg.TOK_EINVAL


def test_product_path_has_no_oracle_dependency():
    # the CUDA library and its binding never import, call or link the oracle
    pkg_dir = os.path.join(ROOT, "exact_bpe_tokenization_utf_gb300")
    for dp, _, fs in os.walk(pkg_dir):
        for f in fs:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".inc")):
                with open(os.path.join(dp, f)) as fh:
                    assert not re.search(r"\boracle\b", fh.read()), f
