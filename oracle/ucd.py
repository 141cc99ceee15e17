"""Code point classes used by the pre-tokenizer patterns.

L  = \\p{L}  (General_Category Lu, Ll, Lt, Lm, Lo)
N  = \\p{N}  (General_Category Nd, Nl, No)
W  = \\s     (the White_Space property: 25 code points)
O  = everything else (marks, symbols, punctuation, controls, unassigned)

The range data in data/unicode_classes.txt was written by
gen_unicode_classes.py from a Unicode regex engine.  TokTier, Section 5.2
(key findings) reports that a Unicode-table version mismatch between two
implementations mis-split about 9,700 code points; the version the data
comes from is recorded in the file's first line.
"""
import bisect
import os

_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "data", "unicode_classes.txt")

_starts, _ends, _cls = [], [], []
with open(_PATH) as _f:
    for _line in _f:
        if _line.startswith("#"):
            continue
        _a, _b, _c = _line.split()
        _starts.append(int(_a, 16))
        _ends.append(int(_b, 16))
        _cls.append(_c)

VERSION_LINE = open(_PATH).readline().strip()

# upper-case and title-case letters (\\p{Lu}, \\p{Lt}): the o200k-style
# pattern splits letter runs by case; data/unicode_upper.txt comes from the
# same generator and regex engine
_UPATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "data", "unicode_upper.txt")
_ustarts, _uends = [], []
with open(_UPATH) as _f:
    for _line in _f:
        if _line.startswith("#"):
            continue
        _a, _b = _line.split()
        _ustarts.append(int(_a, 16))
        _uends.append(int(_b, 16))


# the letters of the CJK scripts (script extensions Han, Hiragana, Katakana,
# Hangul): the DeepSeek-style pattern takes their runs apart from other
# letters; data/unicode_cjk.txt comes from the same generator and regex engine
_CPATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "data", "unicode_cjk.txt")
_cstarts, _cends = [], []
with open(_CPATH) as _f:
    for _line in _f:
        if _line.startswith("#"):
            continue
        _a, _b = _line.split()
        _cstarts.append(int(_a, 16))
        _cends.append(int(_b, 16))


def is_cjk(cp):
    """True for a letter of script extensions Han, Hiragana, Katakana or Hangul."""
    k = bisect.bisect_right(_cstarts, cp) - 1
    return k >= 0 and cp <= _cends[k]


def is_upper(cp):
    """True for an upper-case or title-case letter (Lu, Lt)."""
    k = bisect.bisect_right(_ustarts, cp) - 1
    return k >= 0 and cp <= _uends[k]


def classify(cp):
    """Class letter of one code point."""
    k = bisect.bisect_right(_starts, cp) - 1
    if k >= 0 and cp <= _ends[k]:
        return _cls[k]
    return "O"


def class_array(cps):
    """Class letters of a sequence of code points (memoised per code point)."""
    memo = {}
    out = []
    for cp in cps:
        c = memo.get(cp)
        if c is None:
            c = classify(cp)
            memo[cp] = c
        out.append(c)
    return out
