"""Writes oracle/data/unicode_classes.txt: the code point ranges that the
pre-tokenizer patterns' classes cover.

The patterns are regular expressions, so the authority for what ``\\p{L}``,
``\\p{N}`` and ``\\s`` contain is a Unicode regex engine; this script asks the
third-party ``regex`` module (Unicode tables >= 16.0) about every code point.
Run here, where ``regex`` is installed; the committed output is what the
oracle reads.  Classes: L (letters, General_Category L*), N (numbers, N*),
W (``\\s``, the White_Space property), everything else O.
"""
import os
import sys

import regex


def main(out_path):
    pl, pn, ps = regex.compile(r"\p{L}"), regex.compile(r"\p{N}"), regex.compile(r"\s")
    ranges = []
    cur, start = None, 0
    for cp in range(0x110000 + 1):
        if cp == 0x110000:
            c = None
        elif 0xD800 <= cp <= 0xDFFF:
            c = "O"
        else:
            ch = chr(cp)
            c = "L" if pl.match(ch) else "N" if pn.match(ch) else "W" if ps.match(ch) else "O"
        if c != cur:
            if cur is not None and cur != "O":
                ranges.append((start, cp - 1, cur))
            cur, start = c, cp
    with open(out_path, "w") as f:
        f.write("# regex %s; code point ranges of classes L, N, W (inclusive, hex); others are O\n"
                % regex.__version__)
        for a, b, c in ranges:
            f.write("%04X %04X %s\n" % (a, b, c))
    print(len(ranges), "ranges ->", out_path)


def main_upper(out_path):
    """Ranges of the upper-case letters \\p{Lu} and title-case letters
    \\p{Lt} (the o200k-style pattern's upper-case set)."""
    pu = regex.compile(r"[\p{Lu}\p{Lt}]")
    ranges = []
    start = None
    for cp in range(0x110000 + 1):
        up = cp < 0x110000 and not (0xD800 <= cp <= 0xDFFF) and bool(pu.match(chr(cp)))
        if up and start is None:
            start = cp
        elif not up and start is not None:
            ranges.append((start, cp - 1))
            start = None
    with open(out_path, "w") as f:
        f.write("# regex %s; code point ranges of \\p{Lu} and \\p{Lt} (inclusive, hex)\n" % regex.__version__)
        for a, b in ranges:
            f.write("%04X %04X\n" % (a, b))
    print(len(ranges), "ranges ->", out_path)


# the letters of the CJK scripts: script extensions Han, Hiragana, Katakana or
# Hangul (the DeepSeek-style pattern's CJK runs)
CJK_SET = r"[\p{scx=Han}\p{scx=Hiragana}\p{scx=Katakana}\p{scx=Hangul}]"


def main_cjk(out_path):
    """Ranges of the letters (\\p{L}) whose script extensions include Han,
    Hiragana, Katakana or Hangul."""
    pl, pc = regex.compile(r"\p{L}"), regex.compile(CJK_SET)
    ranges = []
    start = None
    for cp in range(0x110000 + 1):
        ok = cp < 0x110000 and not (0xD800 <= cp <= 0xDFFF) and bool(pl.match(chr(cp))) and bool(pc.match(chr(cp)))
        if ok and start is None:
            start = cp
        elif not ok and start is not None:
            ranges.append((start, cp - 1))
            start = None
    with open(out_path, "w") as f:
        f.write("# regex %s; code point ranges of the letters of script extensions Han, Hiragana, Katakana, "
                "Hangul (inclusive, hex)\n" % regex.__version__)
        for a, b in ranges:
            f.write("%04X %04X\n" % (a, b))
    print(len(ranges), "ranges ->", out_path)


if __name__ == "__main__":
    data = os.path.join(os.path.dirname(os.path.abspath(__file__)), "data")
    main(sys.argv[1] if len(sys.argv) > 1 else os.path.join(data, "unicode_classes.txt"))
    main_upper(sys.argv[2] if len(sys.argv) > 2 else os.path.join(data, "unicode_upper.txt"))
    main_cjk(sys.argv[3] if len(sys.argv) > 3 else os.path.join(data, "unicode_cjk.txt"))
