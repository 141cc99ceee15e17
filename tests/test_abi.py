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


def test_header_compiles_as_c_and_links(libpath, tmp_path):
    # the header is plain C (C99, no warnings); a C program links against the
    # library, reaches every declared entry point, and a load without a usable
    # device is an error code, not a crash
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if not cc:
        pytest.skip("no C compiler")
    syms = declared_symbols()
    src = tmp_path / "abi.c"
    src.write_text("\n".join([
        "#include <stdio.h>",
        '#include "tok.h"',
        "typedef void (*fn)(void);",
        "static const fn entry[] = {" + ", ".join("(fn)%s" % s for s in syms) + "};",
        "int main(void) {",
        "  uint8_t bytes[256]; uint64_t off[257]; tok_handle* h = 0;",
        "  for (int i = 0; i < 256; ++i) { bytes[i] = (uint8_t)i; off[i] = (uint64_t)i; }",
        "  off[256] = 256;",
        "  int rc = tok_load(bytes, off, 256, 0, 0, TOK_PAT_GPT2, &h);",
        "  printf(\"%d %d\\n\", rc, (int)(sizeof entry / sizeof entry[0]));",
        "  if (rc == TOK_OK) tok_free(h);",
        "  return 0;",
        "}",
        ""]))
    exe = tmp_path / "abi"
    libdir = os.path.dirname(libpath)
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"), str(src),
                        "-o", str(exe), "-L", libdir, "-ltokgb", "-Wl,-rpath," + libdir],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    rc, n = (int(x) for x in r.stdout.split())
    assert n == len(syms)
    assert rc in (0, -4)  # TOK_OK with a device, TOK_ECUDA without one
