"""Writes pretoken_pins_o200k.txt: split examples for the o200k-style
pattern, produced by the third-party `regex` module from the pattern text
(the same text include/tok.h and oracle/pretokenize.py state).  The oracle is
checked against these; nothing here calls the oracle or the library.

Run where `regex` is installed:  python tests/golden/make_o200k_pins.py
"""
import json
import os

import regex

O200K_RE = (r"""[^\r\n\p{L}\p{N}]?[\p{Lu}\p{Lt}]*[\p{Ll}\p{Lm}\p{Lo}]+(?:(?i:'s|'t|'re|'ve|'m|'ll|'d))*"""
            r"""|[^\r\n\p{L}\p{N}]?[\p{Lu}\p{Lt}]+(?:(?i:'s|'t|'re|'ve|'m|'ll|'d))*"""
            r"""|\p{N}{1,3}| ?[^\s\p{L}\p{N}]+[\r\n/]*|\s*[\r\n]+|\s+(?!\S)|\s+""")

EXAMPLES = [
    "camelCaseWord", "HTMLParser", "parseHTML", "getXMLHttpRequest", "ABC", "aB", "Ab",
    "don't", "DON'T", "they're here", "we'LL see", "x's", "'s", " 's", "1's", "it'sa", "o'clock", "x'ſ",
    "x's's's", "é'ſ'S", "he'd've", "x'sam's", "'s's", "a''s",
    "中文abc", "abc中文", "ABC中文", "中A", "A中", "中Ab", "ǅungla", "ǅ",
    "x.\n/usr/bin", "a;\r\n/b", ".\n/.abc", "./\n/x", "path/to/file", " //comment\n", "a/\nb", "x\n/y",
    "12345678", "1²3½45", "  foo", "\t\tfoo", "x;\n\n  \ny", "x\r\n\r\n  y", "\n  ", "a.foo", " .foo",
    "IT'S", "'xam", "Hello World", "naïveCafé", "ΑθήναΑθήνα", "éCOLE", "x　y",
]


def main(out):
    rx = regex.compile(O200K_RE)
    with open(out, "w") as f:
        f.write("# o200k-style splits from regex %s; each line: [text, [fragments]]\n" % regex.__version__)
        for s in EXAMPLES:
            f.write(json.dumps([s, rx.findall(s)], ensure_ascii=False) + "\n")
    print(len(EXAMPLES), "pins ->", out)


if __name__ == "__main__":
    main(os.path.join(os.path.dirname(os.path.abspath(__file__)), "pretoken_pins_o200k.txt"))
