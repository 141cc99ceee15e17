"""The CUDA library's code point tables against the oracle's, at every code
point (CPU only: the tables are read from the generated sources).

`ucd_table.inc` (class of a code point: 0 other, 1 letter, 2 number,
3 whitespace) is looked up both ways the kernel does (the two-stage table,
and the direct words below U+10000); `ucd_upper.inc` and `ucd_cjk.inc` are
the o200k-style case bit and the DeepSeek-style CJK-letter bit.  The oracle's
tables come from its own generator (oracle/gen_unicode_classes.py); both
follow the pattern classes \\p{L}, \\p{N}, \\s and \\p{Lu}/\\p{Lt} as the
`regex` module defines them."""
import os
import re

import numpy as np

from oracle.ucd import classify, is_cjk, is_upper

CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                    "exact_bpe_tokenization_utf_gb300", "csrc")
NCP = 0x110000


def _arrays(name):
    text = open(os.path.join(CSRC, name)).read()
    out = {}
    for m in re.finditer(r"(\w+)\[(\d+)\] = \{([^}]*)\}", text):
        vals = [int(v.rstrip("u"), 0) for v in m.group(3).replace("\n", " ").split(",") if v.strip()]
        assert len(vals) == int(m.group(2)), m.group(1)
        out[m.group(1)] = np.array(vals, dtype=np.int64)
    return out


def _oracle(fn):
    return np.array([fn(cp) for cp in range(NCP)], dtype=np.int64)


def test_class_table_both_lookups_match_the_oracle():
    t = _arrays("ucd_table.inc")
    cp = np.arange(NCP, dtype=np.int64)
    two_stage = (t["tok_ucd_stage2"][t["tok_ucd_stage1"][cp >> 8] * 16 + ((cp & 255) >> 4)] >> ((cp & 15) * 2)) & 3
    bmp = cp[:0x10000]
    direct = (t["tok_ucd_bmp"][bmp >> 4] >> ((bmp & 15) * 2)) & 3
    assert np.array_equal(direct, two_stage[:0x10000])
    code = {"O": 0, "L": 1, "N": 2, "W": 3}
    want = _oracle(lambda c: code[classify(c)])
    want[0xD800:0xE000] = 0  # surrogates are never decoded
    assert np.array_equal(two_stage, want)


def _bit_table(name, s1, s2):
    t = _arrays(name)
    cp = np.arange(NCP, dtype=np.int64)
    return (t[s2][t[s1][cp >> 8] * 8 + ((cp & 255) >> 5)] >> (cp & 31)) & 1


def test_upper_and_cjk_bits_match_the_oracle():
    up = _bit_table("ucd_upper.inc", "tok_upper_stage1", "tok_upper_stage2")
    cjk = _bit_table("ucd_cjk.inc", "tok_cjk_stage1", "tok_cjk_stage2")
    assert np.array_equal(up, _oracle(lambda c: int(is_upper(c))))
    assert np.array_equal(cjk, _oracle(lambda c: int(is_cjk(c))))
